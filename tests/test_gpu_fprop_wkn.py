"""GPU parity of Fprop on W's codes as the 128x128 cast stores them, [K x N]
(fp8_block_gemm_fprop_wkn and the FP8BS_OP_FPROP_WKN op of the grouped and
split-K calls): the tensor core reads this operand MN-major. Checked against
the CPU oracle within the GEMM tolerance
    |gpu - oracle| <= 2e-3 * sum_k |a_k b_k| + 1e-6  (+ one BF16 ulp),
and bit for bit against the same GEMM on the byte transpose qT (the same
operand values reach the same tensor-core sums; only their layout in shared
memory differs). Shapes cover several tiles, ragged rows, an output width
that is an odd number of 128-column halves (the last tile's second half
lies wholly past N), stream-K, grouped experts (empty ones included, host
and device offsets) and split-K at long K."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs
import oracle
import workloads as wl
from parity import (absprod_sampled, assert_gemm_close, bf16_values, dequant_blocks, dequant_rows, np_,
                    sample_indices)
from test_gpu_gemm import TILES, q128, q128_oracle, q1x128

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fp8bs.build()
    fp8bs.lib()
    torch.cuda.init()
    yield
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def _both(xq, sx, wq, wqT, sw, M, N):
    y_kn = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_t = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_fprop_wkn(xq, sx, wq, sw, y_kn)
    fp8bs.fp8_block_gemm_fprop(xq, sx, wqT, sw, y_t)
    torch.cuda.synchronize()
    return y_kn, y_t


@pytest.mark.parametrize("M,K,N", [(128, 512, 256), (1, 128, 128), (129, 384, 256), (300, 256, 384),
                                   (257, 1024, 640), (64, 7168, 128), (200, 128, 2304)])
def test_fprop_wkn_small(M, K, N):
    x = wl.with_outliers((M, K), fraction=0.01, seed=M + 3 * K)
    w = wl.normal((K, N), std=wl.W_STD, seed=N + 1)
    xq, sx, oxq, osx = q1x128(x)
    wq, wqT, sw = q128(w)
    owq, osw = q128_oracle(w)
    assert np.array_equal(np_(wq), owq) and np.array_equal(np_(sw), osw)
    y_kn, y_t = _both(xq, sx, wq, wqT, sw, M, N)
    assert torch.equal(y_kn.view(torch.int16), y_t.view(torch.int16)), "MN-major B differs from the transpose"
    ref = oracle.fprop(oxq, osx, owq, osw)
    a, b = dequant_rows(oxq, osx), dequant_blocks(owq, osw)
    assert_gemm_close(bf16_values(y_kn), ref, np.abs(a) @ np.abs(b), True, f"fprop_wkn {M}x{K}x{N}")


def test_fprop_wkn_dense_full():
    """The dense workload (4096 x 7168 x 2048, stream-K on 152 SMs): every
    element equal to the transposed-operand Fprop, samples and whole tiles
    against the oracle."""
    d = wl.dense()
    x, w = d["X"], d["W"]
    xq, sx, oxq, osx = q1x128(x)
    wq, wqT, sw = q128(w)
    owq, osw = q128_oracle(w)
    M, N = x.shape[0], w.shape[1]
    y_kn, y_t = _both(xq, sx, wq, wqT, sw, M, N)
    assert torch.equal(y_kn.view(torch.int16), y_t.view(torch.int16))
    y = bf16_values(y_kn)
    ii, jj = sample_indices(M, N, 32768, seed=3, tiles=TILES)
    ref = oracle.fprop(oxq, osx, owq, osw, ii, jj)
    a = np.abs(dequant_rows(oxq, osx))
    bt = np.ascontiguousarray(np.abs(dequant_blocks(owq, osw)).T)
    assert_gemm_close(y[ii, jj], ref, absprod_sampled(a, bt, ii, jj), True, "fprop_wkn dense full")


def test_fprop_wkn_stream_k():
    """200 output tiles with ragged rows and a half-empty last column tile
    (stream-K on a 152-SM GPU)."""
    M, K, N = 2483, 512, 2432
    x = wl.with_outliers((M, K), fraction=0.01, seed=41)
    w = wl.normal((K, N), std=wl.W_STD, seed=42)
    xq, sx, oxq, osx = q1x128(x)
    wq, wqT, sw = q128(w)
    owq, osw = q128_oracle(w)
    y_kn, y_t = _both(xq, sx, wq, wqT, sw, M, N)
    assert torch.equal(y_kn.view(torch.int16), y_t.view(torch.int16))
    ref = oracle.fprop(oxq, osx, owq, osw)
    bound = np.abs(dequant_rows(oxq, osx)) @ np.abs(dequant_blocks(owq, osw))
    assert_gemm_close(bf16_values(y_kn), ref, bound, True, "fprop_wkn stream-K")


@pytest.mark.parametrize("device_offsets", [False, True])
@pytest.mark.parametrize("counts", [[0, 129, 1, 0, 270], [300, 0], [128, 128, 128]])
def test_grouped_fprop_wkn(counts, device_offsets):
    K, N = 384, 384
    off = wl.offsets_from_counts(counts)
    M, G = int(off[-1]), len(counts)
    x = wl.with_outliers((M, K), fraction=0.01, seed=7 + G)
    w = wl.normal((G, K, N), std=wl.W_STD, seed=8 + G)
    xq, sx, oxq, osx = q1x128(x)
    wq, wqT, sw = q128(w)
    offs = torch.tensor(off, dtype=torch.int32, device="cuda") if device_offsets else off
    y_kn = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_t = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_FPROP_WKN, offs, xq, sx, wq, sw, y_kn, N, K)
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_FPROP, offs, xq, sx, wqT, sw, y_t, N, K)
    torch.cuda.synchronize()
    assert torch.equal(y_kn.view(torch.int16), y_t.view(torch.int16))
    y = bf16_values(y_kn)
    for e in range(G):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        owq, osw = q128_oracle(w[e])
        oxe, osxe = oxq[r0:r1], np.ascontiguousarray(osx[:, r0:r1])
        ref = oracle.fprop(oxe, osxe, owq, osw)
        a, b = dequant_rows(oxe, osxe), dequant_blocks(owq, osw)
        assert_gemm_close(y[r0:r1], ref, np.abs(a) @ np.abs(b), True, f"grouped fprop_wkn e{e}")


@pytest.mark.parametrize("K,splits", [(4096, 8), (16384, 40)])
def test_splitk_fprop_wkn(K, splits):
    M, N = 256, 256
    x = wl.with_outliers((M, K), fraction=0.01, seed=K)
    w = wl.normal((K, N), std=wl.W_STD, seed=K + 1)
    xq, sx, oxq, osx = q1x128(x)
    wq, wqT, sw = q128(w)
    owq, osw = q128_oracle(w)
    outs = []
    for op, b in ((fp8bs.OP_FPROP_WKN, wq), (fp8bs.OP_FPROP, wqT)):
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        fp8bs.fp8_block_gemm_splitk(op, xq, sx, b, sw, out, splits=splits)
        outs.append(out)
    noalloc = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_splitk_noalloc(fp8bs.OP_FPROP_WKN, xq, sx, wq, sw, noalloc, splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.equal(noalloc.view(torch.int16), outs[0].view(torch.int16))
    ii, jj = sample_indices(M, N, 4096, seed=K, tiles=((0, 0), (1, 1)))
    ref = oracle.fprop(oxq, osx, owq, osw, ii, jj)
    a = np.abs(dequant_rows(oxq, osx))
    bt = np.ascontiguousarray(np.abs(dequant_blocks(owq, osw)).T)
    assert_gemm_close(bf16_values(outs[0])[ii, jj], ref, absprod_sampled(a, bt, ii, jj), True,
                      f"split-K fprop_wkn K={K}")


def test_fprop_wkn_rejects_bad_shapes():
    xq = torch.zeros((128, 256), dtype=torch.uint8, device="cuda")
    sx = torch.zeros((2, 128), dtype=torch.float32, device="cuda")
    wq = torch.zeros((256, 200), dtype=torch.uint8, device="cuda")   # N % 128 != 0
    sw = torch.zeros((2, 2), dtype=torch.float32, device="cuda")
    y = torch.empty((128, 200), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8bs.Fp8bsError):
        fp8bs.fp8_block_gemm_fprop_wkn(xq, sx, wq, sw, y)
