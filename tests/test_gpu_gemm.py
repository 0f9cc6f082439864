"""GPU parity of the block-scaled GEMMs (Fprop, Dgrad, Wgrad, grouped) against
the CPU oracle, within the stated tolerance
    |gpu - oracle| <= 2e-3 * sum_k |a_k b_k| + 1e-6  (+ one BF16 ulp for BF16 out).
The operands are quantized on the GPU and checked bit-exact against the
oracle's quantization first, so that both GEMMs consume identical codes.
Small cases compare every output element; the full-size workloads compare
seeded samples plus whole 128x128 output tiles (corners and interior)."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs
import oracle
import workloads as wl
from parity import (absprod_sampled, assert_gemm_close, bf16_values, dequant_blocks,
                    dequant_rows, dequant_tokens_T, np_, sample_indices, u16)

pytestmark = pytest.mark.gpu

TILES = ((0, 0), (-1, -1), (0, -1), (-1, 0), (1, 1), (2, 3), (5, 2), (3, 7))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fp8bs.build()
    fp8bs.lib()
    torch.cuda.init()
    yield
    assert fp8bs.fp8bs_device_status(reset=True) == 0


# ---------------------------------------------------------------------------
# operand preparation on the GPU (checked against the oracle bit for bit)
# ---------------------------------------------------------------------------

def q1x128(x_cpu):
    q, s = fp8bs.empty_quant_1x128(*x_cpu.shape)
    fp8bs.fp8_quant_1x128(x_cpu.cuda(), q, s)
    oq, osc = oracle.quant_1x128(u16(x_cpu))
    R = x_cpu.shape[0]
    assert np.array_equal(np_(q), oq) and np.array_equal(np_(s)[:, :R], osc[:, :R])
    return q, s, oq, osc


def q128(w_cpu):
    batch = w_cpu.shape[0] if w_cpu.dim() == 3 else None
    q, qT, s = fp8bs.empty_quant_128x128(w_cpu.shape[-2], w_cpu.shape[-1], batch=batch)
    fp8bs.fp8_quant_128x128(w_cpu.cuda(), q, qT, s)
    return q, qT, s


def q128_oracle(w_cpu):
    return oracle.quant_128x128(u16(w_cpu))


def requant(src_dev, src_scales, offsets=None):
    qT, scT = fp8bs.empty_requant_128x1_T(src_dev.shape[0], src_dev.shape[1], offsets)
    fp8bs.fp8_requant_128x1_T(src_dev, src_scales, qT, scT, offsets=offsets)
    return qT, scT


# ---------------------------------------------------------------------------
# Fprop
# ---------------------------------------------------------------------------

def run_fprop(x, w):
    xq, sx, oxq, osx = q1x128(x)
    wq, wqT, sw = q128(w)
    owq, osw = q128_oracle(w)
    assert np.array_equal(np_(wq), owq) and np.array_equal(np_(sw), osw)
    y = torch.empty((x.shape[0], w.shape[1]), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_fprop(xq, sx, wqT, sw, y)
    torch.cuda.synchronize()
    return bf16_values(y), (oxq, osx, owq, osw)


@pytest.mark.parametrize("M,K,N", [(128, 512, 256), (1, 128, 128), (129, 384, 256),
                                   (300, 256, 384), (257, 1024, 512), (64, 7168, 128)])
def test_fprop_small(M, K, N):
    x = wl.with_outliers((M, K), fraction=0.01, seed=M + K)
    w = wl.normal((K, N), std=wl.W_STD, seed=N)
    y, (oxq, osx, owq, osw) = run_fprop(x, w)
    ref = oracle.fprop(oxq, osx, owq, osw)
    a = dequant_rows(oxq, osx)
    b = dequant_blocks(owq, osw)
    assert_gemm_close(y, ref, np.abs(a) @ np.abs(b), True, f"fprop {M}x{K}x{N}")


def test_fprop_tiny_workload():
    d = wl.tiny()
    y, (oxq, osx, owq, osw) = run_fprop(d["X"], d["W"])
    ref = oracle.fprop(oxq, osx, owq, osw)
    a, b = dequant_rows(oxq, osx), dequant_blocks(owq, osw)
    assert_gemm_close(y, ref, np.abs(a) @ np.abs(b), True, "fprop tiny")
    # and against the plain fp64 product of the dequantized operands
    assert np.all(np.abs(y - a @ b) <= 2e-3 * (np.abs(a) @ np.abs(b)) + 1e-6 + np.abs(a @ b) * 2 ** -7)


def test_fprop_dense_full_sampled():
    d = wl.dense()
    x, w = d["X"], d["W"]
    y, (oxq, osx, owq, osw) = run_fprop(x, w)
    M, N = y.shape
    ii, jj = sample_indices(M, N, 65536, seed=1, tiles=TILES)
    ref = oracle.fprop(oxq, osx, owq, osw, ii, jj)
    a = np.abs(dequant_rows(oxq, osx))
    bt = np.ascontiguousarray(np.abs(dequant_blocks(owq, osw)).T)
    assert_gemm_close(y[ii, jj], ref, absprod_sampled(a, bt, ii, jj), True, "fprop dense full")


@pytest.mark.parametrize("op", ["fprop", "dgrad"])
def test_stream_k_every_element(op):
    """200 output tiles (ragged rows, a half-empty last column tile) on a
    152-SM GB300: the persistent grid's last round would be a third full,
    so the GEMM runs stream-K, every CTA taking six K-blocks of the
    tile-major sequence and tiles cut between two CTAs finished by the first
    of them. Every element against the oracle; two launches bit-identical."""
    M, C, Wd = 2483, 512, 2432          # rows, contraction, output width
    a_src = wl.with_outliers((M, C), fraction=0.01, seed=41)
    if op == "fprop":
        w = wl.normal((C, Wd), std=wl.W_STD, seed=42)
        y, (oaq, osa, owq, osw) = run_fprop(a_src, w)
        ref = oracle.fprop(oaq, osa, owq, osw)
        bound = np.abs(dequant_rows(oaq, osa)) @ np.abs(dequant_blocks(owq, osw))
        again, _ = run_fprop(a_src, w)
    else:
        w = wl.normal((Wd, C), std=wl.W_STD, seed=43)
        y, (oaq, osa, owq, osw) = run_dgrad(a_src, w)
        ref = oracle.dgrad(oaq, osa, owq, osw)
        bound = np.abs(dequant_rows(oaq, osa)) @ np.abs(dequant_blocks(owq, osw)).T
        again, _ = run_dgrad(a_src, w)
    assert_gemm_close(y, ref, bound, True, f"{op} stream-K {M}x{C}x{Wd}")
    assert np.array_equal(y.view(np.uint32), again.view(np.uint32))


def test_stream_k_on_two_streams_at_once():
    """Two stream-K Fprops issued on two streams with no ordering between
    them each keep their own workspace: both results equal the same GEMMs
    run one after the other."""
    M, K, N = 2483, 512, 2432
    runs = []
    for seed in (51, 52):
        x = wl.with_outliers((M, K), fraction=0.01, seed=seed)
        w = wl.normal((K, N), std=wl.W_STD, seed=seed + 10)
        xq, sx = fp8bs.empty_quant_1x128(M, K)
        fp8bs.fp8_quant_1x128(x.cuda(), xq, sx)
        wq, wqT, sw = fp8bs.empty_quant_128x128(K, N)
        fp8bs.fp8_quant_128x128(w.cuda(), wq, wqT, sw)
        runs.append((xq, sx, wqT, sw))
    torch.cuda.synchronize()
    serial = []
    for xq, sx, wqT, sw in runs:
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        fp8bs.fp8_block_gemm_fprop(xq, sx, wqT, sw, y)
        torch.cuda.synchronize()
        serial.append(y)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:   # each stream's first stream-K GEMM (sets up its workspace)
        with torch.cuda.stream(st):
            xq, sx, wqT, sw = runs[0]
            fp8bs.fp8_block_gemm_fprop(xq, sx, wqT, sw, torch.empty((M, N), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in runs]
    for _ in range(4):
        for st, (xq, sx, wqT, sw), y in zip(streams, runs, outs):
            with torch.cuda.stream(st):
                fp8bs.fp8_block_gemm_fprop(xq, sx, wqT, sw, y)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    for y, ref in zip(outs, serial):
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("K", [128, 384])
def test_stream_k_short_contraction(K):
    """Stream-K with one and three K-blocks per tile (200 tiles of 128 x 256:
    ranges of two and four K-blocks, so with three per tile most tiles are
    cut, some at their first K-block). Every element against the oracle."""
    M, N = 12745, 512
    x = wl.with_outliers((M, K), fraction=0.01, seed=K + 5)
    w = wl.normal((K, N), std=wl.W_STD, seed=K + 6)
    y, (oxq, osx, owq, osw) = run_fprop(x, w)
    ref = oracle.fprop(oxq, osx, owq, osw)
    bound = np.abs(dequant_rows(oxq, osx)) @ np.abs(dequant_blocks(owq, osw))
    assert_gemm_close(y, ref, bound, True, f"fprop stream-K {M}x{K}x{N}")


@pytest.mark.parametrize("op", ["fprop", "fprop_wkn", "dgrad"])
def test_grouped_many_tiles_host_and_device_offsets(op):
    """220 output tiles of 128 x 256 over six experts (empty ones included),
    two K-blocks each, more tiles than a 152-SM GPU's persistent grid: host
    and device offsets give the same bytes, and every expert's rows match
    the oracle."""
    counts = [0, 300, 129, 1, 0, 2000]
    off = wl.offsets_from_counts(counts)
    M, G = int(off[-1]), len(counts)
    C, Wd = 256, 2432                     # contraction, output width
    a_src = wl.with_outliers((M, C), fraction=0.01, seed=71)
    aq, sa, oaq, osa = q1x128(a_src)
    if op == "dgrad":
        w = wl.normal((G, Wd, C), std=wl.W_STD, seed=72)    # W_e [K = Wd x N = C]
        wq, _, sw = q128(w)
        b, N, K, opc = wq, C, Wd, fp8bs.OP_DGRAD
    else:
        w = wl.normal((G, C, Wd), std=wl.W_STD, seed=73)    # W_e [K = C x N = Wd]
        wq, wqT, sw = q128(w)
        b, N, K = (wqT, Wd, C) if op == "fprop" else (wq, Wd, C)
        opc = fp8bs.OP_FPROP if op == "fprop" else fp8bs.OP_FPROP_WKN
    outs = []
    for offs in (off, torch.tensor(off, dtype=torch.int32, device="cuda")):
        y = torch.full((M, Wd), float("nan"), dtype=torch.bfloat16, device="cuda")
        fp8bs.fp8_block_gemm_grouped(opc, offs, aq, sa, b, sw, y, N, K)
        outs.append(y)
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    y = bf16_values(outs[0])
    for e in range(G):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        owq, osw = q128_oracle(w[e])
        oae, osae = oaq[r0:r1], np.ascontiguousarray(osa[:, r0:r1])
        a = np.abs(dequant_rows(oae, osae))
        bb = np.abs(dequant_blocks(owq, osw))
        if op == "dgrad":
            ref, bound = oracle.dgrad(oae, osae, owq, osw), a @ bb.T
        else:
            ref, bound = oracle.fprop(oae, osae, owq, osw), a @ bb
        assert_gemm_close(y[r0:r1], ref, bound, True, f"grouped many tiles {op} e{e}")


# ---------------------------------------------------------------------------
# Dgrad
# ---------------------------------------------------------------------------

def run_dgrad(dy, w):
    dyq, sdy, odyq, osdy = q1x128(dy)
    wq, _, sw = q128(w)
    owq, osw = q128_oracle(w)
    dx = torch.empty((dy.shape[0], w.shape[0]), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_dgrad(dyq, sdy, wq, sw, dx)
    torch.cuda.synchronize()
    return bf16_values(dx), (odyq, osdy, owq, osw)


@pytest.mark.parametrize("M,N,K", [(128, 256, 512), (1, 128, 128), (129, 384, 256),
                                   (300, 2048, 384), (200, 128, 640)])
def test_dgrad_small(M, N, K):
    dy = wl.with_outliers((M, N), fraction=0.01, seed=M + N + 1)
    w = wl.normal((K, N), std=wl.W_STD, seed=K)
    dx, (odyq, osdy, owq, osw) = run_dgrad(dy, w)
    ref = oracle.dgrad(odyq, osdy, owq, osw)
    a, b = dequant_rows(odyq, osdy), dequant_blocks(owq, osw)
    assert_gemm_close(dx, ref, np.abs(a) @ np.abs(b).T, True, f"dgrad {M}x{N}x{K}")


def test_dgrad_zero_rows_are_exactly_zero():
    """Leading zero rows and sparse non-zero rows of dY give exactly zero dX rows."""
    M, N, K = 300, 256, 384
    dy = wl.normal((M, N), std=wl.DY_STD, seed=4)
    dy[:40] = 0.0
    keep = torch.zeros(M, dtype=torch.bool)
    keep[::17] = True
    dy[~keep & (torch.arange(M) >= 40)] = 0.0
    w = wl.normal((K, N), std=wl.W_STD, seed=5)
    dx, _ = run_dgrad(dy, w)
    zero_rows = (dy.float().abs().sum(1) == 0).numpy()
    assert zero_rows.sum() > 200
    assert np.all(dx[zero_rows] == 0.0)
    assert np.all(np.isfinite(dx))


def test_dgrad_backward_full_sampled():
    d = wl.backward()
    dx, (odyq, osdy, owq, osw) = run_dgrad(d["dY"], d["W"])
    M, K = dx.shape
    ii, kk = sample_indices(M, K, 65536, seed=2, tiles=TILES)
    ref = oracle.dgrad(odyq, osdy, owq, osw, ii, kk)
    a = np.abs(dequant_rows(odyq, osdy))
    b = np.abs(dequant_blocks(owq, osw))
    assert_gemm_close(dx[ii, kk], ref, absprod_sampled(a, b, ii, kk), True, "dgrad backward full")


# ---------------------------------------------------------------------------
# Wgrad
# ---------------------------------------------------------------------------

def run_wgrad(dy, x, x_from_stash=True, accumulate_into=None):
    """dW = dY^T X with dY requantized from BF16 and X from its E4M3 stash."""
    dyT, sdyT = requant(dy.cuda(), None)
    if x_from_stash:
        xq, sx, _, _ = q1x128(x)
        xT, sxT = requant(xq, sx)
    else:
        xT, sxT = requant(x.cuda(), None)
    N, K = dy.shape[1], x.shape[1]
    if accumulate_into is None:
        dw = torch.full((N, K), float("nan"), dtype=torch.float32, device="cuda")
        fp8bs.fp8_block_gemm_wgrad(dyT, sdyT, xT, sxT, dw)
    else:
        dw = accumulate_into.clone().cuda()
        fp8bs.fp8_block_gemm_wgrad(dyT, sdyT, xT, sxT, dw, accumulate=True)
    torch.cuda.synchronize()
    return np_(dw), (np_(dyT), np_(sdyT), np_(xT), np_(sxT))


def _oracle_wgrad_operands(dy, x, x_from_stash=True):
    odyT, osdyT = oracle.requant_128x1_T(u16(dy))
    if x_from_stash:
        oxq, osx = oracle.quant_1x128(u16(x))
        oxT, osxT = oracle.requant_128x1_T(oxq, osx)
    else:
        oxT, osxT = oracle.requant_128x1_T(u16(x))
    return odyT, osdyT, oxT, osxT


@pytest.mark.parametrize("T,N,K,stash", [(128, 128, 256, True), (300, 256, 128, True),
                                         (1, 128, 128, False), (513, 384, 512, False),
                                         (1000, 128, 1024, True)])
def test_wgrad_small(T, N, K, stash):
    dy = wl.with_outliers((T, N), fraction=0.01, seed=T + N)
    x = wl.with_outliers((T, K), fraction=0.01, seed=T + K + 1)
    dw, ops = run_wgrad(dy, x, stash)
    odyT, osdyT, oxT, osxT = _oracle_wgrad_operands(dy, x, stash)
    for g_, o_ in zip(ops, (odyT, osdyT, oxT, osxT)):
        assert np.array_equal(g_, o_)
    ref = oracle.wgrad(odyT, osdyT, oxT, osxT)
    a, b = dequant_tokens_T(odyT, osdyT), dequant_tokens_T(oxT, osxT)
    assert_gemm_close(dw, ref, np.abs(a) @ np.abs(b).T, False, f"wgrad {T}x{N}x{K}")


def test_wgrad_accumulate():
    T, N, K = 256, 128, 256
    dy = wl.normal((T, N), seed=1)
    x = wl.normal((T, K), seed=2)
    base = wl.normal((N, K), seed=3).float()
    dw, _ = run_wgrad(dy, x, accumulate_into=base)
    dw0, _ = run_wgrad(dy, x)
    assert np.allclose(dw, dw0 + base.numpy(), rtol=1e-6, atol=1e-6)


def test_wgrad_all_zero_grad_is_exactly_zero():
    T, N, K = 384, 256, 256
    dy = torch.zeros((T, N), dtype=torch.bfloat16)
    x = wl.normal((T, K), seed=7)
    dw, _ = run_wgrad(dy, x)
    assert np.all(dw == 0.0)


def test_wgrad_backward_full_sampled():
    d = wl.backward()
    dw, ops = run_wgrad(d["dY"], d["X"])
    odyT, osdyT, oxT, osxT = _oracle_wgrad_operands(d["dY"], d["X"])
    for g_, o_ in zip(ops, (odyT, osdyT, oxT, osxT)):
        assert np.array_equal(g_, o_)
    N, K = dw.shape
    nn, kk = sample_indices(N, K, 65536, seed=3, tiles=TILES)
    ref = oracle.wgrad(odyT, osdyT, oxT, osxT, nn, kk)
    a = np.abs(dequant_tokens_T(odyT, osdyT))
    b = np.abs(dequant_tokens_T(oxT, osxT))
    assert_gemm_close(dw[nn, kk], ref, absprod_sampled(a, b, nn, kk), False, "wgrad backward full")


# ---------------------------------------------------------------------------
# Grouped (MoE experts)
# ---------------------------------------------------------------------------

def _grouped_case(counts, K, N, seed):
    off = wl.offsets_from_counts(counts)
    M = int(off[-1])
    G = len(counts)
    x = wl.with_outliers((M, K), fraction=0.01, seed=seed)
    w = wl.normal((G, K, N), std=wl.W_STD, seed=seed + 1)
    return off, x, w


@pytest.mark.parametrize("counts", [[0, 129, 1, 0, 270], [5], [300, 0], [128, 128, 128]])
def test_grouped_fprop_small(counts):
    K, N = 256, 384
    off, x, w = _grouped_case(counts, K, N, seed=len(counts))
    xq, sx, oxq, osx = q1x128(x)
    wq, wqT, sw = q128(w)
    y = torch.full((x.shape[0], N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_FPROP, off, xq, sx, wqT, sw, y, N, K)
    torch.cuda.synchronize()
    y = bf16_values(y)
    for e in range(len(counts)):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        owq, osw = q128_oracle(w[e])
        oxe, osxe = oxq[r0:r1], np.ascontiguousarray(osx[:, r0:r1])
        ref = oracle.fprop(oxe, osxe, owq, osw)
        a, b = dequant_rows(oxe, osxe), dequant_blocks(owq, osw)
        assert_gemm_close(y[r0:r1], ref, np.abs(a) @ np.abs(b), True, f"grouped fprop e{e}")


@pytest.mark.parametrize("counts", [[0, 129, 1, 0, 270], [300, 0]])
def test_grouped_dgrad_small(counts):
    N, K = 384, 256       # dgrad contracts over N, writes K columns
    off = wl.offsets_from_counts(counts)
    M, G = int(off[-1]), len(counts)
    dy = wl.with_outliers((M, N), fraction=0.01, seed=11)
    w = wl.normal((G, K, N), std=wl.W_STD, seed=12)
    dyq, sdy, odyq, osdy = q1x128(dy)
    wq, _, sw = q128(w)
    dx = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_DGRAD, off, dyq, sdy, wq, sw, dx, N, K)
    torch.cuda.synchronize()
    dx = bf16_values(dx)
    for e in range(G):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        owq, osw = q128_oracle(w[e])
        oe, ose = odyq[r0:r1], np.ascontiguousarray(osdy[:, r0:r1])
        ref = oracle.dgrad(oe, ose, owq, osw)
        a, b = dequant_rows(oe, ose), dequant_blocks(owq, osw)
        assert_gemm_close(dx[r0:r1], ref, np.abs(a) @ np.abs(b).T, True, f"grouped dgrad e{e}")


@pytest.mark.parametrize("counts", [[0, 129, 1, 0, 270], [128], [0, 0]])
def test_grouped_wgrad_small(counts):
    N, K = 256, 384
    off = wl.offsets_from_counts(counts)
    M, G = int(off[-1]), len(counts)
    dy = wl.with_outliers((M, N), fraction=0.01, seed=21)
    a_ = wl.with_outliers((M, K), fraction=0.01, seed=22)
    dyT, sdyT = requant(dy.cuda(), None, off)
    aT, saT = requant(a_.cuda(), None, off)
    dw = torch.full((G, N, K), float("nan"), dtype=torch.float32, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_WGRAD, off, dyT, sdyT, aT, saT, dw, N, K)
    torch.cuda.synchronize()
    dw = np_(dw)
    odyT, osdyT = oracle.requant_128x1_T(u16(dy), offsets=off)
    oaT, osaT = oracle.requant_128x1_T(u16(a_), offsets=off)
    assert np.array_equal(np_(dyT), odyT) and np.array_equal(np_(aT), oaT)
    p = 0
    for e in range(G):
        n_e = int(off[e + 1] - off[e])
        w_e = -(-n_e // 128) * 128
        if n_e == 0:
            assert np.all(dw[e] == 0.0)       # empty expert: exactly zero gradient
            continue
        ref = oracle.wgrad(odyT, osdyT, oaT, osaT, t0=p, t1=p + w_e)
        a = dequant_tokens_T(odyT[:, p:p + w_e], osdyT[p // 128:(p + w_e) // 128])
        b = dequant_tokens_T(oaT[:, p:p + w_e], osaT[p // 128:(p + w_e) // 128])
        assert_gemm_close(dw[e], ref, np.abs(a) @ np.abs(b).T, False, f"grouped wgrad e{e}")
        p += w_e


@pytest.mark.slow
def test_grouped_moe_full_sampled():
    """The MoE workload at full size: up-projection Fprop, down-projection
    Fprop, Dgrad and Wgrad, each checked on sampled elements of a few experts."""
    d = wl.moe()
    off, counts = d["offsets"], d["counts"]
    G = len(counts)
    hidden, inter, up = 7168, 2048, 4096
    nonempty = [e for e in range(G) if counts[e] > 0]
    check = sorted(set([nonempty[0], nonempty[-1], int(np.argmax(counts)), nonempty[len(nonempty) // 2]]))
    rng = np.random.default_rng(5)

    # up projection: Y = X W_up_e, W_up_e [hidden x up]
    xq, sx, oxq, osx = q1x128(d["X"])
    wq, wqT, sw = q128(d["W_up"])
    y = torch.empty((8192, up), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_FPROP, off, xq, sx, wqT, sw, y, up, hidden)
    # down projection fprop: Y = A W_down_e, W_down_e [inter x hidden]
    aq, sa, oaq, osa = q1x128(d["A"])
    wdq, wdqT, swd = q128(d["W_down"])
    y2 = torch.empty((8192, hidden), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_FPROP, off, aq, sa, wdqT, swd, y2, hidden, inter)
    # down projection dgrad: dA = dY W_down_e^T
    dyq, sdy, odyq, osdy = q1x128(d["dY"])
    da = torch.empty((8192, inter), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_DGRAD, off, dyq, sdy, wdq, swd, da, hidden, inter)
    # down projection wgrad: dW_e = dY_e^T A_e
    dyT, sdyT = requant(d["dY"].cuda(), None, off)
    aT, saT = requant(aq, sa, off)
    dw = torch.empty((G, hidden, inter), dtype=torch.float32, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_WGRAD, off, dyT, sdyT, aT, saT, dw, hidden, inter)
    torch.cuda.synchronize()
    y, y2, da, dw = bf16_values(y), bf16_values(y2), bf16_values(da), np_(dw)
    odyT, osdyT = oracle.requant_128x1_T(u16(d["dY"]), offsets=off)
    oaT, osaT = oracle.requant_128x1_T(oaq, osa, offsets=off)
    assert np.array_equal(np_(dyT), odyT) and np.array_equal(np_(aT), oaT)
    pstarts = np.concatenate([[0], np.cumsum(-(-counts // 128) * 128)])

    for e in check:
        r0, r1 = int(off[e]), int(off[e + 1])
        n = 2048
        rows = rng.integers(r0, r1, n)
        # up fprop
        owq, osw = q128_oracle(d["W_up"][e])
        cols = rng.integers(0, up, n)
        oxe, osxe = oxq[r0:r1], np.ascontiguousarray(osx[:, r0:r1])
        ref = oracle.fprop(oxe, osxe, owq, osw, rows - r0, cols)
        a = np.abs(dequant_rows(oxe, osxe))[rows - r0]
        b = np.abs(dequant_blocks(owq, osw))[:, cols]
        assert_gemm_close(y[rows, cols], ref, np.einsum("ek,ke->e", a, b), True, f"moe up e{e}")
        # down fprop
        owdq, oswd = q128_oracle(d["W_down"][e])
        cols = rng.integers(0, hidden, n)
        oae, osae = oaq[r0:r1], np.ascontiguousarray(osa[:, r0:r1])
        ref = oracle.fprop(oae, osae, owdq, oswd, rows - r0, cols)
        a = np.abs(dequant_rows(oae, osae))[rows - r0]
        b = np.abs(dequant_blocks(owdq, oswd))[:, cols]
        assert_gemm_close(y2[rows, cols], ref, np.einsum("ek,ke->e", a, b), True, f"moe down e{e}")
        # down dgrad
        cols = rng.integers(0, inter, n)
        ode, osde = odyq[r0:r1], np.ascontiguousarray(osdy[:, r0:r1])
        ref = oracle.dgrad(ode, osde, owdq, oswd, rows - r0, cols)
        a = np.abs(dequant_rows(ode, osde))[rows - r0]
        b = np.abs(dequant_blocks(owdq, oswd))[cols]
        assert_gemm_close(da[rows, cols], ref, np.einsum("en,en->e", a, b), True, f"moe dgrad e{e}")
        # down wgrad
        p0, p1 = int(pstarts[e]), int(pstarts[e + 1])
        nn, kk = rng.integers(0, hidden, n), rng.integers(0, inter, n)
        ref = oracle.wgrad(odyT, osdyT, oaT, osaT, nn, kk, t0=p0, t1=p1)
        a = np.abs(dequant_tokens_T(odyT[:, p0:p1], osdyT[p0 // 128:p1 // 128]))[nn]
        b = np.abs(dequant_tokens_T(oaT[:, p0:p1], osaT[p0 // 128:p1 // 128]))[kk]
        assert_gemm_close(dw[e][nn, kk], ref, np.einsum("et,et->e", a, b), False, f"moe wgrad e{e}")
    for e in range(G):
        if counts[e] == 0:
            assert np.all(dw[e] == 0.0)


# ---------------------------------------------------------------------------
# Long-K drift workload
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("K", wl.LONGK_VALUES)
def test_longk_promoted_error_stays_flat(K):
    d = wl.longk(K)
    y, (oxq, osx, owq, osw) = run_fprop(d["X"], d["W"])
    ii, jj = sample_indices(256, 256, 512, seed=K, tiles=((0, 0),))
    ref = oracle.fprop(oxq, osx, owq, osw, ii, jj)
    truth, _ = oracle.fprop_reference_sums(oxq, osx, owq, osw, ii, jj, unpromoted=False)
    absprod = np.abs(truth)  # all operands positive: sum |a b| = |sum a b|
    assert_gemm_close(y[ii, jj], ref, absprod, True, f"longk {K}")
    rel = np.abs(y[ii, jj] - truth) / np.abs(truth)
    assert rel.max() < 2 ** -7   # within BF16 output rounding of the fp64 truth


def test_gemm_outputs_are_deterministic():
    x = wl.normal((300, 512), seed=1)
    w = wl.normal((512, 256), std=wl.W_STD, seed=2)
    y1, _ = run_fprop(x, w)
    y2, _ = run_fprop(x, w)
    assert np.array_equal(y1, y2)
