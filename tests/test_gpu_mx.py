"""GPU parity of the MXFP8 path against the oracle: the 1x32
quantizer byte for byte (codes and exponent bytes, read back from the scale
atoms), and the hardware block-scaled GEMM within the GEMM tolerance
|d| <= 2e-3 * sum_k |a_k b_k| + 1e-6 plus one BF16 ulp."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs
import oracle
import workloads as wl
from parity import assert_gemm_close, bf16_values, np_, sample_indices, u16
from test_gpu_quant import _special_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fp8bs.build()
    fp8bs.lib()
    torch.cuda.init()
    yield
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def atoms_to_rows(atoms: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Exponent bytes [rows x cols/32] from the scale-atom layout."""
    kb = cols // 128
    a = atoms[: (rows + 127) // 128 * kb * 512].reshape(-1, kb, 32, 4, 4)   # [r128][kb][m0][m1][j]
    a = a.transpose(0, 3, 2, 1, 4).reshape(-1, kb * 4)                      # row = 128 r128 + 32 m1 + m0
    return a[:rows]


def mx_quant(x_cpu):
    R, C = x_cpu.shape
    q, at = fp8bs.empty_mx_quant(R, C)
    fp8bs.fp8_mx_quant_1x32(x_cpu.cuda(), q, at)
    torch.cuda.synchronize()
    return q, at


@pytest.mark.parametrize("R,C", [(1, 128), (5, 256), (300, 384), (129, 1024)])
def test_mx_quant_matches_oracle(R, C):
    x = _special_inputs(R, C, seed=R * 3 + C)
    q, at = mx_quant(x)
    oq, oe = oracle.mx_quant_1x32(u16(x))
    assert np.array_equal(np_(q), oq)
    assert np.array_equal(atoms_to_rows(np_(at), R, C), oe)
    pad = atoms_to_rows(np_(at), (R + 127) // 128 * 128, C)[R:]
    assert np.all(pad == 127)


def _dequant(q, e):
    t = oracle.e4m3_table().astype(np.float64)
    return t[q] * np.repeat(np.ldexp(1.0, e.astype(np.int64) - 127), 32, 1)


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 256, 512), (1, 512, 256), (257, 768, 1024)])
def test_mx_gemm_small(M, N, K):
    a = wl.with_outliers((M, K), fraction=0.01, seed=M + K)
    b = wl.normal((N, K), std=wl.W_STD, seed=N + K)
    qa, aa = mx_quant(a)
    qb, ab = mx_quant(b)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_mx_gemm(qa, aa, qb, ab, out)
    torch.cuda.synchronize()
    oqa, oea = oracle.mx_quant_1x32(u16(a))
    oqb, oeb = oracle.mx_quant_1x32(u16(b))
    ref = oracle.mx_gemm(oqa, oea, oqb, oeb)
    absprod = np.abs(_dequant(oqa, oea)) @ np.abs(_dequant(oqb, oeb)).T
    assert_gemm_close(bf16_values(out), ref, absprod, True, f"mx gemm {M}x{N}x{K}")


def test_mx_gemm_dense_fprop_sampled():
    """The dense layer's Fprop in MXFP8: X 4096x7168, W^T 2048x7168."""
    d = wl.dense()
    x, wt = d["X"], d["W"].t().contiguous()
    qa, aa = mx_quant(x)
    qb, ab = mx_quant(wt)
    out = torch.empty((4096, 2048), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_mx_gemm(qa, aa, qb, ab, out)
    torch.cuda.synchronize()
    oqa, oea = oracle.mx_quant_1x32(u16(x))
    oqb, oeb = oracle.mx_quant_1x32(u16(wt))
    assert np.array_equal(np_(qa), oqa) and np.array_equal(np_(qb), oqb)
    ii, jj = sample_indices(4096, 2048, 8192, seed=3, tiles=((0, 0), (-1, -1)))
    ref = oracle.mx_gemm(oqa, oea, oqb, oeb, ii, jj)
    da, db = np.abs(_dequant(oqa, oea)), np.abs(_dequant(oqb, oeb))
    absprod = np.einsum("ek,ek->e", da[ii], db[jj])
    assert_gemm_close(bf16_values(out)[ii, jj], ref, absprod, True, "mx dense fprop")


def _pad_rows(x_cpu, mult=128):
    R, C = x_cpu.shape
    rp = (R + mult - 1) // mult * mult
    out = torch.zeros((rp, C), dtype=x_cpu.dtype)
    out[:R] = x_cpu
    return out


def mx_quant_T(x_cpu):
    R, C = x_cpu.shape
    qT, at = fp8bs.empty_mx_quant_T(R, C)
    fp8bs.fp8_mx_quant_1x32_T(x_cpu.cuda(), qT, at)
    torch.cuda.synchronize()
    return qT, at


@pytest.mark.parametrize("R,C", [(128, 128), (300, 256), (1, 16), (129, 144), (257, 400)])
def test_mx_quant_T_matches_oracle_of_transpose(R, C):
    """The transposed MXFP8 cast equals the oracle's 1x32 cast of the
    zero-padded transpose: codes (padding tokens 0x00), exponent bytes, and
    127 in the atoms' padding rows."""
    x = _special_inputs(R, C, seed=R * 7 + C)
    qT, at = mx_quant_T(x)
    xt = _pad_rows(x).t().contiguous()                      # [C x Mpad]
    Mp = xt.shape[1]
    oq, oe = oracle.mx_quant_1x32(u16(xt))
    assert np.array_equal(np_(qT), oq)
    assert np.array_equal(atoms_to_rows(np_(at), C, Mp), oe)
    pad = atoms_to_rows(np_(at), (C + 127) // 128 * 128, Mp)[C:]
    assert np.all(pad == 127)


def test_mx_quant_T_backward_dy_full():
    dy = wl.backward()["dY"]                                # 4096 x 2048
    qT, at = mx_quant_T(dy)
    oq, oe = oracle.mx_quant_1x32(u16(dy.t().contiguous()))
    assert np.array_equal(np_(qT), oq)
    assert np.array_equal(atoms_to_rows(np_(at), dy.shape[1], dy.shape[0]), oe)


def _mx_ref(a_q, a_e, b_q, b_e, ii=None, jj=None):
    ref = oracle.mx_gemm(a_q, a_e, b_q, b_e, ii, jj)
    da, db = np.abs(_dequant(a_q, a_e)), np.abs(_dequant(b_q, b_e))
    absprod = da @ db.T if ii is None else np.einsum("ek,ek->e", da[ii], db[jj])
    return ref, absprod


@pytest.mark.parametrize("T,N,K", [(128, 128, 256), (300, 256, 512), (1, 128, 256)])
def test_mx_wgrad_f32(T, N, K):
    """MXFP8 Wgrad dW [N x K] = dY^T X in FP32, both operands from the
    transposed cast (32-token blocks), against the oracle's MX GEMM of the
    oracle's casts of the padded transposes."""
    dy = wl.normal((T, N), std=wl.DY_STD, seed=T + N)
    x = wl.with_outliers((T, K), fraction=0.01, seed=T + K)
    qa, aa = mx_quant_T(dy)
    qb, ab = mx_quant_T(x)
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    fp8bs.fp8_mx_gemm_f32(qa, aa, qb, ab, out)
    torch.cuda.synchronize()
    oqa, oea = oracle.mx_quant_1x32(u16(_pad_rows(dy).t().contiguous()))
    oqb, oeb = oracle.mx_quant_1x32(u16(_pad_rows(x).t().contiguous()))
    assert np.array_equal(np_(qa), oqa) and np.array_equal(np_(qb), oqb)
    ref, absprod = _mx_ref(oqa, oea, oqb, oeb)
    assert_gemm_close(np_(out), ref, absprod, False, f"mx wgrad {T}x{N}x{K}")


def test_mx_dgrad_small():
    """MXFP8 Dgrad dX [M x K] = dY W: A = the 1x32 cast of dY along N, B =
    the 1x32 cast of W [K x N] along N."""
    M, N, K = 300, 256, 512
    dy = wl.normal((M, N), std=wl.DY_STD, seed=11)
    w = wl.normal((K, N), std=wl.W_STD, seed=12)
    qa, aa = mx_quant(dy)
    qb, ab = mx_quant(w)
    out = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_mx_gemm(qa, aa, qb, ab, out)
    torch.cuda.synchronize()
    oqa, oea = oracle.mx_quant_1x32(u16(dy))
    oqb, oeb = oracle.mx_quant_1x32(u16(w))
    ref, absprod = _mx_ref(oqa, oea, oqb, oeb)
    assert_gemm_close(bf16_values(out), ref, absprod, True, "mx dgrad")


def test_mx_fprop_with_transposed_weight_cast():
    """MXFP8 Fprop Y = X W with B = the transposed cast of W [K x N] (no BF16
    transpose of W needed)."""
    M, K, N = 257, 512, 256
    x = wl.with_outliers((M, K), fraction=0.01, seed=21)
    w = wl.normal((K, N), std=wl.W_STD, seed=22)
    qa, aa = mx_quant(x)
    qb, ab = mx_quant_T(w)                                  # [N x K]
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_mx_gemm(qa, aa, qb, ab, out)
    torch.cuda.synchronize()
    oqa, oea = oracle.mx_quant_1x32(u16(x))
    oqb, oeb = oracle.mx_quant_1x32(u16(w.t().contiguous()))
    assert np.array_equal(np_(qb), oqb)
    ref, absprod = _mx_ref(oqa, oea, oqb, oeb)
    assert_gemm_close(bf16_values(out), ref, absprod, True, "mx fprop, transposed W cast")


def test_mx_wgrad_dense_sampled():
    """The dense layer's Wgrad in MXFP8 (T = 4096, dW 2048 x 7168), sampled."""
    d = wl.backward()
    dy, x = d["dY"], d["X"]
    qa, aa = mx_quant_T(dy)
    qb, ab = mx_quant_T(x)
    out = torch.empty((2048, 7168), dtype=torch.float32, device="cuda")
    fp8bs.fp8_mx_gemm_f32(qa, aa, qb, ab, out)
    torch.cuda.synchronize()
    oqa, oea = oracle.mx_quant_1x32(u16(dy.t().contiguous()))
    oqb, oeb = oracle.mx_quant_1x32(u16(x.t().contiguous()))
    ii, jj = sample_indices(2048, 7168, 4096, seed=5, tiles=((0, 0), (-1, -1)))
    ref, absprod = _mx_ref(oqa, oea, oqb, oeb, ii, jj)
    assert_gemm_close(np_(out)[ii, jj], ref, absprod, False, "mx dense wgrad")


# ---------------------------------------------------------------------------
# The tensor core's own accumulation over the whole contraction (config 5's
# "unpromoted" counterpart on this GPU): the MX GEMM keeps one tensor-memory
# accumulator over all of K, with the power-of-two block scales applied
# inside the MMA, and no software promotion.
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K", wl.LONGK_VALUES)
def test_hardware_accumulation_over_long_k(K):
    """Long-K drift workload (X 256xK, W Kx256, U(0.5, 1.5): same-sign
    products, so accumulation errors add up). Against the fp64 sum over the
    dequantized MX operands, the FP32-output MX GEMM's relative error stays
    within the worst-case bound of an fp32 accumulator over K positive terms,
    (K - 1) 2^-24, whatever the order of the additions (E4M3 products and
    power-of-two scalings are exact in fp32). The drift model of "FP8 动态量化
    里的 partial sum 漂移", section 4, with a 14-bit accumulator (the oracle's
    unpromoted sum of the 1x128 / 128x128 operands) drifts far past that
    bound at long K; the hardware accumulator does not."""
    d = wl.longk(K)
    x, wt = d["X"], d["W"].t().contiguous()
    qa, aa = mx_quant(x)
    qb, ab = mx_quant(wt)
    out = torch.empty((256, 256), dtype=torch.float32, device="cuda")
    fp8bs.fp8_mx_gemm_f32(qa, aa, qb, ab, out)
    torch.cuda.synchronize()
    oqa, oea = oracle.mx_quant_1x32(u16(x))
    oqb, oeb = oracle.mx_quant_1x32(u16(wt))
    ii, jj = sample_indices(256, 256, 256, seed=K)
    A = _dequant(oqa[np.unique(ii)], oea[np.unique(ii)])
    B = _dequant(oqb[np.unique(jj)], oeb[np.unique(jj)])
    ia = {r: n for n, r in enumerate(np.unique(ii))}
    jb = {c: n for n, c in enumerate(np.unique(jj))}
    truth = np.array([A[ia[i]] @ B[jb[j]] for i, j in zip(ii, jj)])
    got = np_(out)[ii, jj].astype(np.float64)
    rel_hw = np.abs(got - truth) / truth
    assert rel_hw.max() <= (K - 1) * 2.0 ** -24, f"K={K}: hardware accumulation rel err {rel_hw.max():.3e}"
    # the drift model's 14-bit unpromoted accumulation on the same workload
    xq, sx = oracle.quant_1x128(u16(d["X"]))
    wq, sw = oracle.quant_128x128(u16(d["W"]))
    t64, u14 = oracle.fprop_reference_sums(xq, sx, wq, sw, ii[:64], jj[:64], m_bits=14)
    rel_14 = np.abs(u14 - t64) / t64
    print(f"K={K}: hardware fp32 accumulation max rel err {rel_hw.max():.3e} "
          f"(bound {(K - 1) * 2.0 ** -24:.3e}); 14-bit unpromoted model {rel_14.max():.3e}")
    if K >= 16384:
        assert rel_14.max() > (K - 1) * 2.0 ** -24 > rel_hw.max()
