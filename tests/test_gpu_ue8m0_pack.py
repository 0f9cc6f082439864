"""GPU parity of the packed Blackwell scale layout for power-of-two scales:
fp8_pack_ue8m0 byte for byte against the oracle's packing (read
back from the scale atoms) for the four operand layouts, the error it
records for a scale without an exponent byte, and the recipe's three GEMMs
run through the MX kernel on packed UE8M0 operands against the oracle's
promoted GEMMs within |d| <= 2e-3 * sum_k |a_k b_k| + 1e-6 (plus one BF16
ulp for BF16 outputs)."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs
import oracle
import workloads as wl
from parity import assert_gemm_close, bf16_values, np_
from test_gpu_mx import atoms_to_rows

pytestmark = pytest.mark.gpu

UE8M0 = fp8bs.ScaleOpts(fp8bs.SCALE_UE8M0, 0.0, 0.0)
FP8BS_ERR_DEVICE = 7


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fp8bs.build()
    fp8bs.lib()
    torch.cuda.init()
    yield
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def _operands(M, K, N, seed):
    """UE8M0-rule casts on the GPU of X [M x K], W [K x N], dY [M x N]."""
    x = wl.with_outliers((M, K), fraction=0.01, seed=seed)
    w = wl.normal((K, N), std=wl.W_STD, seed=seed + 1)
    dy = wl.normal((M, N), std=wl.DY_STD, seed=seed + 2)
    xq, sx = fp8bs.empty_quant_1x128(M, K)
    fp8bs.fp8_quant_1x128_opts(x.cuda(), xq, sx, UE8M0)
    wq, wqT, sw = fp8bs.empty_quant_128x128(K, N)
    fp8bs.fp8_quant_128x128_opts(w.cuda(), wq, wqT, sw, UE8M0)
    dyq, sdy = fp8bs.empty_quant_1x128(M, N)
    dyT, sdyT = fp8bs.empty_requant_128x1_T(M, N)
    fp8bs.fp8_quant_dual_opts(dy.cuda(), dyq, sdy, dyT, sdyT, UE8M0)
    xT, sxT = fp8bs.empty_requant_128x1_T(M, K)
    fp8bs.fp8_requant_128x1_T_opts(xq, sx, xT, sxT, UE8M0)
    torch.cuda.synchronize()
    return dict(xq=xq, sx=sx, wq=wq, wqT=wqT, sw=sw, dyq=dyq, sdy=sdy, dyT=dyT, sdyT=sdyT, xT=xT, sxT=sxT)


def _pack(scales, rows, K, row_block, row_stride, kb_stride):
    atoms = torch.full((fp8bs.fp8bs_mx_scale_bytes(rows, K),), 0xEE, dtype=torch.uint8, device="cuda")
    fp8bs.fp8_pack_ue8m0(scales, rows, K, row_block, row_stride, kb_stride, atoms)
    torch.cuda.synchronize()
    return atoms


def _layouts(d, M, K, N):
    """(name, scales, rows, contraction, row_block, row_stride, kb_stride) of
    the six operands of Fprop, Dgrad and Wgrad."""
    Mp = d["xT"].shape[1]
    return [
        ("X rows", d["sx"], M, K, 1, 1, d["sx"].shape[1]),
        ("W^T (Fprop B)", d["sw"], N, K, 128, 1, N // 128),
        ("dY rows", d["sdy"], M, N, 1, 1, d["sdy"].shape[1]),
        ("W (Dgrad B)", d["sw"], K, N, 128, N // 128, 1),
        ("dY^T (Wgrad A)", d["sdyT"], N, Mp, 1, 1, N),
        ("X^T (Wgrad B)", d["sxT"], K, Mp, 1, 1, K),
    ]


@pytest.mark.parametrize("M,K,N", [(200, 384, 256), (1, 256, 128), (513, 512, 384)])
def test_pack_matches_oracle(M, K, N):
    d = _operands(M, K, N, seed=M + K)
    for name, sc, rows, contr, rb, rs, ks in _layouts(d, M, K, N):
        atoms = np_(_pack(sc, rows, contr, rb, rs, ks))
        ref, bad = oracle.pack_ue8m0(np_(sc), rows, contr, rb, rs, ks)
        assert bad == 0, name
        assert np.array_equal(atoms_to_rows(atoms, rows, contr), ref), name
        pad = atoms_to_rows(atoms, (rows + 127) // 128 * 128, contr)[rows:]
        assert np.all(pad == 127), name
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def test_pack_records_scales_without_an_exponent_byte():
    """A scale that is not a power of two (0.75), zero, or out of range
    (2^-130) gets byte 255 and the device status FP8BS_ERR_DEVICE; the
    others keep their bytes."""
    rows, K = 130, 256
    s = np.ones((2, 132), np.float32)
    s[0, 3], s[1, 7], s[0, 129] = 0.75, 0.0, 2.0 ** -130
    s[1, 5] = 2.0 ** -20
    atoms = np_(_pack(torch.from_numpy(s).cuda(), rows, K, 1, 1, 132))
    assert fp8bs.fp8bs_device_status(reset=True) == FP8BS_ERR_DEVICE
    got = atoms_to_rows(atoms, rows, K)
    ref, bad = oracle.pack_ue8m0(s, rows, K, 1, 1, 132)
    assert bad == 3 and np.array_equal(got, ref)
    assert (got[3, :4] == 255).all() and (got[7, 4:] == 255).all() and (got[129, :4] == 255).all()
    assert (got[5, 4:] == 107).all()


@pytest.mark.parametrize("M,K,N", [(200, 512, 256), (300, 768, 512)])
def test_ue8m0_gemms_through_the_mx_kernel(M, K, N):
    """Fprop, Dgrad and Wgrad of UE8M0-rule operands run by the MX GEMM on
    packed scales, against the oracle's promoted GEMMs on the same codes and
    scales."""
    d = _operands(M, K, N, seed=7 * M + N)
    lay = {name: _pack(sc, rows, contr, rb, rs, ks) for name, sc, rows, contr, rb, rs, ks in _layouts(d, M, K, N)}
    h = {k: np_(v) for k, v in d.items()}
    dec = lambda q: oracle.e4m3_decode(q).astype(np.float64)

    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_mx_gemm(d["xq"], lay["X rows"], d["wqT"], lay["W^T (Fprop B)"], y)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_mx_gemm(d["dyq"], lay["dY rows"], d["wq"], lay["W (Dgrad B)"], dx)
    dw = torch.empty((N, K), dtype=torch.float32, device="cuda")
    fp8bs.fp8_mx_gemm_f32(d["dyT"], lay["dY^T (Wgrad A)"], d["xT"], lay["X^T (Wgrad B)"], dw)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0

    xa = np.abs(dec(h["xq"]) * np.repeat(h["sx"][:, :M].T, 128, axis=1))
    wa = np.abs(dec(h["wq"]) * np.repeat(np.repeat(h["sw"], 128, axis=0), 128, axis=1))
    da = np.abs(dec(h["dyq"]) * np.repeat(h["sdy"][:, :M].T, 128, axis=1))
    assert_gemm_close(bf16_values(y), oracle.fprop(h["xq"], h["sx"], h["wq"], h["sw"]), xa @ wa, True,
                      f"ue8m0 fprop {M}x{K}x{N}")
    assert_gemm_close(bf16_values(dx), oracle.dgrad(h["dyq"], h["sdy"], h["wq"], h["sw"]), da @ wa.T, True,
                      f"ue8m0 dgrad {M}x{N}x{K}")
    dta = np.abs(dec(h["dyT"]) * np.repeat(h["sdyT"].T, 128, axis=1))    # [N x Mpad]
    xta = np.abs(dec(h["xT"]) * np.repeat(h["sxT"].T, 128, axis=1))      # [K x Mpad]
    assert_gemm_close(np_(dw), oracle.wgrad(h["dyT"], h["sdyT"], h["xT"], h["sxT"]), dta @ xta.T, False,
                      f"ue8m0 wgrad {M}: {N}x{K}")


@pytest.mark.parametrize("M,K,N", [(200, 512, 256), (129, 256, 768), (300, 1024, 512)])
def test_mx_fprop_on_w_as_stored(M, K, N):
    """The MX Fprop on W's codes [K x N] (fp8_mx_gemm_wkn: the tensor core
    reads them MN-major, with the W^T atoms) equals the MX Fprop on the byte
    transpose bit for bit, and the packed weight cast without the transpose
    writes the same codes, scales and atoms; the result is within the GEMM
    tolerance of the oracle's promoted Fprop on the same codes."""
    x = wl.with_outliers((M, K), fraction=0.01, seed=M + K)
    w = wl.normal((K, N), std=wl.W_STD, seed=N + 5)
    xq, sx = fp8bs.empty_quant_1x128(M, K)
    fp8bs.fp8_quant_1x128_opts(x.cuda(), xq, sx, UE8M0)
    ax = _pack(sx, M, K, 1, 1, sx.shape[1])
    wd = w.cuda()
    wq, wqT, sw = fp8bs.empty_quant_128x128(K, N)
    awT, aw = fp8bs.empty_mx_atoms(N, K), fp8bs.empty_mx_atoms(K, N)
    fp8bs.fp8_quant_128x128_packed(wd, wq, wqT, sw, awT, aw)
    wq2, _, sw2 = fp8bs.empty_quant_128x128(K, N, with_transpose=False)
    awT2, aw2 = fp8bs.empty_mx_atoms(N, K), fp8bs.empty_mx_atoms(K, N)
    fp8bs.fp8_quant_128x128_packed(wd, wq2, None, sw2, awT2, aw2)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    y2 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_mx_gemm(xq, ax, wqT, awT, y)
    fp8bs.fp8_mx_gemm_wkn(xq, ax, wq2, awT2, y2)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    for a, b in ((wq, wq2), (sw, sw2), (awT, awT2), (aw, aw2)):
        assert torch.equal(a, b)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    h = {k: np_(v) for k, v in dict(xq=xq, sx=sx, wq=wq, sw=sw).items()}
    dec = lambda q: oracle.e4m3_decode(q).astype(np.float64)
    xa = np.abs(dec(h["xq"]) * np.repeat(h["sx"][:, :M].T, 128, axis=1))
    wa = np.abs(dec(h["wq"]) * np.repeat(np.repeat(h["sw"], 128, axis=0), 128, axis=1))
    assert_gemm_close(bf16_values(y2), oracle.fprop(h["xq"], h["sx"], h["wq"], h["sw"]), xa @ wa, True,
                      f"mx fprop on W [K x N] {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N,batch", [(200, 384, 256, 1), (513, 512, 384, 1), (128, 256, 128, 3)])
def test_packed_casts_equal_cast_then_pack(M, K, N, batch):
    """The casts that write their scale atoms in the same pass give the same
    codes and scales as the UE8M0 casts, and the same atoms as
    fp8_pack_ue8m0 of those scales (and as the oracle's packing)."""
    x = wl.with_outliers((M, K), fraction=0.01, seed=M)
    dy = wl.normal((M, N), std=wl.DY_STD, seed=M + 1)
    w = wl.normal((batch, K, N) if batch > 1 else (K, N), std=wl.W_STD, seed=M + 2).cuda()
    Mp = fp8bs.fp8bs_padded_tokens(M)
    # weights
    wq, wqT, sw = fp8bs.empty_quant_128x128(K, N, batch=batch)
    fp8bs.fp8_quant_128x128_opts(w, wq, wqT, sw, UE8M0)
    pq, pqT, psw = fp8bs.empty_quant_128x128(K, N, batch=batch)
    aT, aW = fp8bs.empty_mx_atoms(N, K, batch), fp8bs.empty_mx_atoms(K, N, batch)
    fp8bs.fp8_quant_128x128_packed(w, pq, pqT, psw, aT, aW)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    assert torch.equal(wq, pq) and torch.equal(wqT, pqT) and torch.equal(sw, psw)
    nb = fp8bs.fp8bs_mx_scale_bytes(N, K)
    for b in range(batch):
        swb = sw.view(batch, -1)[b].contiguous()
        assert torch.equal(aT[b * nb:(b + 1) * nb], _pack(swb, N, K, 128, 1, N // 128)), b
        assert torch.equal(aW[b * nb:(b + 1) * nb], _pack(swb, K, N, 128, N // 128, 1)), b
        ref, bad = oracle.pack_ue8m0(np_(swb), N, K, 128, 1, N // 128)
        assert bad == 0 and np.array_equal(atoms_to_rows(np_(aT[b * nb:(b + 1) * nb]), N, K), ref)
    # activations (stash) and gradients (dual)
    for name, src, C in (("stash", x, K), ("dual", dy, N)):
        q, s = fp8bs.empty_quant_1x128(M, C)
        qT, sT = fp8bs.empty_requant_128x1_T(M, C)
        (fp8bs.fp8_quant_dual_stash_opts if name == "stash" else fp8bs.fp8_quant_dual_opts)(
            src.cuda(), q, s, qT, sT, UE8M0)
        pq, ps = fp8bs.empty_quant_1x128(M, C)
        pqT, psT = fp8bs.empty_requant_128x1_T(M, C)
        aq, aqT = fp8bs.empty_mx_atoms(M, C), fp8bs.empty_mx_atoms(C, Mp)
        (fp8bs.fp8_quant_dual_stash_packed if name == "stash" else fp8bs.fp8_quant_dual_packed)(
            src.cuda(), pq, ps, pqT, psT, aq, aqT)
        torch.cuda.synchronize()
        assert fp8bs.fp8bs_device_status(reset=True) == 0, name
        # (the scale array's columns past row M are padding that no cast writes)
        for a, b in ((q, pq), (s[:, :M], ps[:, :M]), (qT, pqT), (sT, psT)):
            assert torch.equal(a, b), name
        assert torch.equal(aq, _pack(s, M, C, 1, 1, s.shape[1])), name
        assert torch.equal(aqT, _pack(sT, C, Mp, 1, 1, C)), name
        ref, bad = oracle.pack_ue8m0(np_(s), M, C, 1, 1, s.shape[1])
        assert bad == 0 and np.array_equal(atoms_to_rows(np_(aq), M, C), ref), name
        assert np.all(atoms_to_rows(np_(aq), (M + 127) // 128 * 128, C)[M:] == 127), name


def test_packed_cast_flags_a_scale_without_a_byte():
    """A row tile of tiny values has a UE8M0 scale below 2^-127: the fused
    cast writes byte 255 for it and records FP8BS_ERR_DEVICE, as the
    separate packing does."""
    M, C = 128, 256
    x = wl.normal((M, C), std=1.0, seed=9)
    x[5, 128:] = 1.0e-38                       # BF16 subnormal; amax / 448 far below 2^-127
    q, s = fp8bs.empty_quant_1x128(M, C)
    qT, sT = fp8bs.empty_requant_128x1_T(M, C)
    aq, aqT = fp8bs.empty_mx_atoms(M, C), fp8bs.empty_mx_atoms(C, M)
    fp8bs.fp8_quant_dual_packed(x.cuda(), q, s, qT, sT, aq, aqT)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == FP8BS_ERR_DEVICE
    got = atoms_to_rows(np_(aq), M, C)
    ref, bad = oracle.pack_ue8m0(np_(s), M, C, 1, 1, s.shape[1])
    assert bad == 1 and np.array_equal(got, ref)
    assert (got[5, 4:] == 255).all() and (got[5, :4] != 255).all()
