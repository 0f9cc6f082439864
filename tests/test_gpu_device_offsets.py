"""Grouped (MoE) calls with DEVICE group offsets, and the stream-ordered
status calls.

With offsets in device memory the kernels derive each group's rows, tiles and
padded token segment when they run, so the MoE pass needs no host copy of
the routing and can be one captured CUDA graph whose routing changes between
replays. Checked here:
  - the transposed, dual and fused casts and the three grouped GEMMs with
    device offsets give bytes identical to the same calls with host offsets
    (which the oracle parity tests cover), on ragged groups with empty
    experts; the capacity columns past the groups' padded total are left
    untouched; one case of each is also compared with the oracle directly;
  - the whole MoE pass (the MoE workload at full size) captured once in a
    graph with device offsets, replayed under two different routings, matches
    the oracle on sampled elements of several experts and is byte-identical
    to eager host-offset calls;
  - invalid device offsets record FP8BS_ERR_DEVICE (read stream-ordered) and
    write nothing, and the context stays usable.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs
import oracle
import workloads as wl
from parity import (assert_gemm_close, bf16_values, dequant_blocks, dequant_rows, dequant_tokens_T, np_, u16)

pytestmark = pytest.mark.gpu

ERR_DEVICE, ERR_TIMEOUT = 7, 5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fp8bs.build()
    fp8bs.lib()
    torch.cuda.init()
    yield
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def _dev(off):
    return torch.tensor(np.asarray(off, np.int32), dtype=torch.int32, device="cuda")


def _bits(t):
    return np_(t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.uint8))


def _raw(t):
    """Bit patterns of any tensor (fp32 as uint32)."""
    return np_(t).view(np.uint32) if t.dtype == torch.float32 else _bits(t)


COUNTS = [[0, 129, 1, 0, 270], [300, 0], [5], [0, 0, 128, 0]]


@pytest.mark.parametrize("counts", COUNTS)
def test_transposed_casts_device_offsets_match_host_offsets(counts):
    off = wl.offsets_from_counts(counts)
    M, C, G = int(off[-1]), 256, len(counts)
    x = wl.with_outliers((M, C), fraction=0.01, seed=40 + G)
    xd = x.cuda()
    offd = _dev(off)
    mp = fp8bs.fp8bs_padded_tokens(M, off)
    cap = fp8bs.fp8bs_padded_tokens_max(M, G)
    assert mp <= cap
    xq, sx = fp8bs.empty_quant_1x128(M, C)
    fp8bs.fp8_quant_1x128(xd, xq, sx)
    for name, call in (
            ("requant B", lambda o, qT, sT, q, s: fp8bs.fp8_requant_128x1_T(xd, None, qT, sT, offsets=o)),
            ("requant Q", lambda o, qT, sT, q, s: fp8bs.fp8_requant_128x1_T(xq, sx, qT, sT, offsets=o)),
            ("dual", lambda o, qT, sT, q, s: fp8bs.fp8_quant_dual(xd, q, s, qT, sT, offsets=o)),
            ("stash", lambda o, qT, sT, q, s: fp8bs.fp8_quant_dual_stash(xd, q, s, qT, sT, offsets=o))):
        hT, hs = fp8bs.empty_requant_128x1_T(M, C, off)
        hq, hsc = fp8bs.empty_quant_1x128(M, C)
        call(off, hT, hs, hq, hsc)
        dT = torch.full((C, cap), 0xA5, dtype=torch.uint8, device="cuda")
        ds = torch.full((cap // 128, C), -7.0, dtype=torch.float32, device="cuda")
        dq, dsc = fp8bs.empty_quant_1x128(M, C)
        assert dT.shape == fp8bs.empty_requant_128x1_T(M, C, offd)[0].shape
        call(offd, dT, ds, dq, dsc)
        torch.cuda.synchronize()
        assert np.array_equal(np_(dT)[:, :mp], np_(hT)), name
        assert np.array_equal(np_(ds)[:mp // 128], np_(hs)), name
        assert np.all(np_(dT)[:, mp:] == 0xA5) and np.all(np_(ds)[mp // 128:] == -7.0), name
        if name in ("dual", "stash"):
            assert np.array_equal(np_(dq), np_(hq)) and np.array_equal(np_(dsc)[:, :M], np_(hsc)[:, :M]), name
    # and directly against the oracle (BF16 source)
    oT, os_ = oracle.requant_128x1_T(u16(x), offsets=off)
    dT = torch.empty((C, cap), dtype=torch.uint8, device="cuda")
    ds = torch.empty((cap // 128, C), dtype=torch.float32, device="cuda")
    fp8bs.fp8_requant_128x1_T_dev(xd, None, dT, ds, offd)
    torch.cuda.synchronize()
    assert np.array_equal(np_(dT)[:, :mp], oT) and np.array_equal(np_(ds)[:mp // 128], os_)
    assert fp8bs.fp8bs_last_device_status(reset=True) == 0


@pytest.mark.parametrize("counts", COUNTS)
def test_grouped_gemms_device_offsets_match_host_offsets(counts):
    off = wl.offsets_from_counts(counts)
    M, G = int(off[-1]), len(counts)
    K, N = 256, 384
    offd = _dev(off)
    x = wl.with_outliers((M, K), fraction=0.01, seed=50 + G)
    w = wl.normal((G, K, N), std=wl.W_STD, seed=51)
    dy = wl.with_outliers((M, N), fraction=0.01, seed=52)
    xq, sx = fp8bs.empty_quant_1x128(M, K)
    fp8bs.fp8_quant_1x128(x.cuda(), xq, sx)
    dyq, sdy = fp8bs.empty_quant_1x128(M, N)
    fp8bs.fp8_quant_1x128(dy.cuda(), dyq, sdy)
    wq, wqT, sw = fp8bs.empty_quant_128x128(K, N, batch=G)
    fp8bs.fp8_quant_128x128(w.cuda(), wq, wqT, sw)
    # Fprop and Dgrad
    for op, a, sa, b, width in ((fp8bs.OP_FPROP, xq, sx, wqT, N), (fp8bs.OP_DGRAD, dyq, sdy, wq, K)):
        yh = torch.full((M, width), float("nan"), dtype=torch.bfloat16, device="cuda")
        yd = torch.full((M, width), float("nan"), dtype=torch.bfloat16, device="cuda")
        fp8bs.fp8_block_gemm_grouped(op, off, a, sa, b, sw, yh, N, K)
        fp8bs.fp8_block_gemm_grouped(op, offd, a, sa, b, sw, yd, N, K)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(yd), _bits(yh)), op
    # Wgrad on the capacity layout of the device-offset casts
    cap = fp8bs.fp8bs_padded_tokens_max(M, G)
    dyT, sdyT = fp8bs.empty_requant_128x1_T(M, N, offd)
    xT, sxT = fp8bs.empty_requant_128x1_T(M, K, offd)
    fp8bs.fp8_requant_128x1_T(dy.cuda(), None, dyT, sdyT, offsets=offd)
    fp8bs.fp8_requant_128x1_T(xq, sx, xT, sxT, offsets=offd)
    assert dyT.shape == (N, cap)
    dwd = torch.full((G, N, K), float("nan"), dtype=torch.float32, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_WGRAD, offd, dyT, sdyT, xT, sxT, dwd, N, K, rows=M)
    hdyT, hsdyT = fp8bs.empty_requant_128x1_T(M, N, off)
    hxT, hsxT = fp8bs.empty_requant_128x1_T(M, K, off)
    fp8bs.fp8_requant_128x1_T(dy.cuda(), None, hdyT, hsdyT, offsets=off)
    fp8bs.fp8_requant_128x1_T(xq, sx, hxT, hsxT, offsets=off)
    dwh = torch.full((G, N, K), float("nan"), dtype=torch.float32, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_WGRAD, off, hdyT, hsdyT, hxT, hsxT, dwh, N, K)
    torch.cuda.synchronize()
    assert np.array_equal(np_(dwd).view(np.uint32), np_(dwh).view(np.uint32))
    # against the oracle: Wgrad per expert (exact zeros for empty experts)
    oxq, osx = oracle.quant_1x128(u16(x))
    odyT, osdyT = oracle.requant_128x1_T(u16(dy), offsets=off)
    oxT, osxT = oracle.requant_128x1_T(oxq, osx, offsets=off)
    dw = np_(dwd)
    p = 0
    for e in range(G):
        n_e = int(off[e + 1] - off[e])
        w_e = -(-n_e // 128) * 128
        if n_e == 0:
            assert np.all(dw[e] == 0.0)
            continue
        ref = oracle.wgrad(odyT, osdyT, oxT, osxT, t0=p, t1=p + w_e)
        a = dequant_tokens_T(odyT[:, p:p + w_e], osdyT[p // 128:(p + w_e) // 128])
        b = dequant_tokens_T(oxT[:, p:p + w_e], osxT[p // 128:(p + w_e) // 128])
        assert_gemm_close(dw[e], ref, np.abs(a) @ np.abs(b).T, False, f"device-offset wgrad e{e}")
        p += w_e
    assert fp8bs.fp8bs_last_device_status(reset=True) == 0


@pytest.mark.parametrize("bad", [[1, 129, 130, 300], [0, 200, 100, 300], [0, 100, 200, 299]])
def test_invalid_device_offsets_record_error_and_write_nothing(bad):
    """off[0] != 0, a decrease, a total other than rows: FP8BS_ERR_DEVICE in
    the status word (read in stream order), no output written, and the next
    call with valid offsets is correct."""
    M, C, K, N, G = 300, 256, 256, 384, 3
    offd = _dev(bad)
    x = wl.normal((M, C), seed=60).cuda()
    qT, sT = fp8bs.empty_requant_128x1_T(M, C, offd)
    qT.fill_(0x5A)
    assert fp8bs.fp8bs_last_device_status(reset=True) == 0
    fp8bs.fp8_requant_128x1_T(x, None, qT, sT, offsets=offd)
    assert fp8bs.fp8bs_last_device_status(reset=True) == ERR_DEVICE
    assert np.all(np_(qT) == 0x5A)
    for fn in (fp8bs.fp8_quant_dual, fp8bs.fp8_quant_dual_stash):   # the grouped tile kernel
        q, s = fp8bs.empty_quant_1x128(M, C)
        q.fill_(0x5A)
        fn(x, q, s, qT, sT, offsets=offd)
        assert fp8bs.fp8bs_last_device_status(reset=True) == ERR_DEVICE, fn.__name__
        assert np.all(np_(qT) == 0x5A) and np.all(np_(q) == 0x5A), fn.__name__
    xq, sx = fp8bs.empty_quant_1x128(M, K)
    fp8bs.fp8_quant_1x128(wl.normal((M, K), seed=61).cuda(), xq, sx)
    wq, wqT, sw = fp8bs.empty_quant_128x128(K, N, batch=G)
    fp8bs.fp8_quant_128x128(wl.normal((G, K, N), std=wl.W_STD, seed=62).cuda(), wq, wqT, sw)
    y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_FPROP, offd, xq, sx, wqT, sw, y, N, K)
    assert fp8bs.fp8bs_last_device_status(reset=True) == ERR_DEVICE
    assert torch.all(y == 3.0)
    good = wl.offsets_from_counts([100, 0, 200])
    yh = torch.empty_like(y)
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_FPROP, good, xq, sx, wqT, sw, yh, N, K)
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_FPROP, _dev(good), xq, sx, wqT, sw, y, N, K)
    assert fp8bs.fp8bs_last_device_status(reset=True) == 0
    assert torch.equal(y.view(torch.int16), yh.view(torch.int16))


def test_stream_ordered_status_calls():
    """fp8bs_last_device_status waits for its stream only and reports the
    status as of the work issued on it; fp8bs_copy_device_status copies the
    word into a device tensor without waiting (and can reset it)."""
    s = torch.cuda.Stream()
    assert fp8bs.fp8bs_last_device_status(s, reset=True) == 0
    with torch.cuda.stream(s):
        fp8bs.fp8bs_selftest_wait_timeout(2_000_000)          # 2 ms wait that gives up
    assert fp8bs.fp8bs_last_device_status(s) == ERR_TIMEOUT   # still set: no reset
    dst = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    fp8bs.fp8bs_copy_device_status(dst, reset=True, stream=s)
    s.synchronize()
    assert int(dst.item()) == ERR_TIMEOUT
    assert fp8bs.fp8bs_last_device_status(s) == 0
    dst.fill_(-1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fp8bs.fp8bs_copy_device_status(dst)
    graph.replay()
    torch.cuda.synchronize()
    assert int(dst.item()) == 0


def _moe_outputs(G, cap, dev="cuda"):
    hidden, inter, up, M = 7168, 2048, 4096, 8192
    o = {}
    o["xq"], o["sx"] = fp8bs.empty_quant_1x128(M, hidden)
    o["aq"], o["sa"] = fp8bs.empty_quant_1x128(M, inter)
    o["dyq"], o["sdy"] = fp8bs.empty_quant_1x128(M, hidden)
    o["aT"] = torch.empty((inter, cap), dtype=torch.uint8, device=dev)
    o["saT"] = torch.empty((cap // 128, inter), dtype=torch.float32, device=dev)
    o["dyT"] = torch.empty((hidden, cap), dtype=torch.uint8, device=dev)
    o["sdyT"] = torch.empty((cap // 128, hidden), dtype=torch.float32, device=dev)
    o["y"] = torch.empty((M, up), dtype=torch.bfloat16, device=dev)
    o["y2"] = torch.empty((M, hidden), dtype=torch.bfloat16, device=dev)
    o["da"] = torch.empty((M, inter), dtype=torch.bfloat16, device=dev)
    o["dw"] = torch.empty((G, hidden, inter), dtype=torch.float32, device=dev)
    return o


def _moe_pass(o, offsets, inp, W, w_as_stored=False):
    """The routed part of the MoE pass: the casts of X, of the down-projection
    input A (with the 128x1 requant of its stash) and of dY (both
    orientations), the up and down Fprop (on the weights' transposed codes,
    or with w_as_stored on their codes as stored, read MN-major), the down
    Dgrad and Wgrad."""
    hidden, inter, up, M = 7168, 2048, 4096, 8192
    fprop, wu, wd = ((fp8bs.OP_FPROP_WKN, W["wuq"], W["wdq"]) if w_as_stored
                     else (fp8bs.OP_FPROP, W["wuqT"], W["wdqT"]))
    fp8bs.fp8_quant_1x128(inp["X"], o["xq"], o["sx"])
    fp8bs.fp8_quant_dual_stash(inp["A"], o["aq"], o["sa"], o["aT"], o["saT"], offsets=offsets)
    fp8bs.fp8_quant_dual(inp["dY"], o["dyq"], o["sdy"], o["dyT"], o["sdyT"], offsets=offsets)
    fp8bs.fp8_block_gemm_grouped(fprop, offsets, o["xq"], o["sx"], wu, W["swu"], o["y"], up, hidden)
    fp8bs.fp8_block_gemm_grouped(fprop, offsets, o["aq"], o["sa"], wd, W["swd"], o["y2"], hidden, inter)
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_DGRAD, offsets, o["dyq"], o["sdy"], W["wdq"], W["swd"], o["da"],
                                 hidden, inter)
    fp8bs.fp8_block_gemm_grouped(fp8bs.OP_WGRAD, offsets, o["dyT"], o["sdyT"], o["aT"], o["saT"], o["dw"],
                                 hidden, inter, rows=M)


def _check_moe_against_oracle(o, d, off, W_cpu, experts, seed):
    """Sampled elements of the four GEMMs of `experts` against the oracle."""
    counts = np.diff(off)
    hidden, inter, up = 7168, 2048, 4096
    rng = np.random.default_rng(seed)
    oxq, osx = oracle.quant_1x128(u16(d["X"]))
    oaq, osa = oracle.quant_1x128(u16(d["A"]))
    odyq, osdy = oracle.quant_1x128(u16(d["dY"]))
    assert np.array_equal(np_(o["xq"]), oxq) and np.array_equal(np_(o["aq"]), oaq)
    odyT, osdyT = oracle.requant_128x1_T(u16(d["dY"]), offsets=off)
    oaT, osaT = oracle.requant_128x1_T(oaq, osa, offsets=off)
    mp = odyT.shape[1]
    assert np.array_equal(np_(o["dyT"])[:, :mp], odyT) and np.array_equal(np_(o["aT"])[:, :mp], oaT)
    y, y2, da, dw = bf16_values(o["y"]), bf16_values(o["y2"]), bf16_values(o["da"]), np_(o["dw"])
    pstarts = np.concatenate([[0], np.cumsum(-(-counts // 128) * 128)])
    n = 1024
    for e in experts:
        r0, r1 = int(off[e]), int(off[e + 1])
        rows = rng.integers(r0, r1, n)
        owq, osw = oracle.quant_128x128(u16(W_cpu["W_up"][e]))
        cols = rng.integers(0, up, n)
        oxe, osxe = oxq[r0:r1], np.ascontiguousarray(osx[:, r0:r1])
        ref = oracle.fprop(oxe, osxe, owq, osw, rows - r0, cols)
        a = np.abs(dequant_rows(oxe, osxe))[rows - r0]
        b = np.abs(dequant_blocks(owq, osw))[:, cols]
        assert_gemm_close(y[rows, cols], ref, np.einsum("ek,ke->e", a, b), True, f"graph moe up e{e}")
        owdq, oswd = oracle.quant_128x128(u16(W_cpu["W_down"][e]))
        cols = rng.integers(0, hidden, n)
        oae, osae = oaq[r0:r1], np.ascontiguousarray(osa[:, r0:r1])
        ref = oracle.fprop(oae, osae, owdq, oswd, rows - r0, cols)
        a = np.abs(dequant_rows(oae, osae))[rows - r0]
        b = np.abs(dequant_blocks(owdq, oswd))[:, cols]
        assert_gemm_close(y2[rows, cols], ref, np.einsum("ek,ke->e", a, b), True, f"graph moe down e{e}")
        cols = rng.integers(0, inter, n)
        ode, osde = odyq[r0:r1], np.ascontiguousarray(osdy[:, r0:r1])
        ref = oracle.dgrad(ode, osde, owdq, oswd, rows - r0, cols)
        a = np.abs(dequant_rows(ode, osde))[rows - r0]
        b = np.abs(dequant_blocks(owdq, oswd))[cols]
        assert_gemm_close(da[rows, cols], ref, np.einsum("en,en->e", a, b), True, f"graph moe dgrad e{e}")
        p0, p1 = int(pstarts[e]), int(pstarts[e + 1])
        nn, kk = rng.integers(0, hidden, n), rng.integers(0, inter, n)
        ref = oracle.wgrad(odyT, osdyT, oaT, osaT, nn, kk, t0=p0, t1=p1)
        a = np.abs(dequant_tokens_T(odyT[:, p0:p1], osdyT[p0 // 128:p1 // 128]))[nn]
        b = np.abs(dequant_tokens_T(oaT[:, p0:p1], osaT[p0 // 128:p1 // 128]))[kk]
        assert_gemm_close(dw[e][nn, kk], ref, np.einsum("et,et->e", a, b), False, f"graph moe wgrad e{e}")
    for e in range(len(counts)):
        if counts[e] == 0:
            assert np.all(dw[e] == 0.0)


@pytest.mark.slow
def test_moe_pass_one_graph_device_offsets_two_routings():
    """The MoE workload's routed pass captured ONCE as a CUDA graph that reads
    its offsets from device memory, its Fprops on the experts' weight codes
    as stored (the benchmarked form); replayed under the workload's routing
    and under a second routing written into the same offsets tensor. Each
    replay is byte-identical to eager calls with host offsets and the
    transposed weight codes, and matches the oracle on sampled elements of
    several experts (empty experts: exact zero dW)."""
    d = wl.moe()
    G, M = len(d["counts"]), 8192
    off1 = d["offsets"]
    c2 = np.random.default_rng(77).multinomial(M, np.random.default_rng(78).dirichlet([0.5] * G))
    off2 = wl.offsets_from_counts(c2)
    assert not np.array_equal(off1, off2)
    inp = {k: d[k].cuda() for k in ("X", "A", "dY")}
    W = {}
    W["wuq"], W["wuqT"], W["swu"] = fp8bs.empty_quant_128x128(7168, 4096, batch=G)
    fp8bs.fp8_quant_128x128(d["W_up"].cuda(), W["wuq"], W["wuqT"], W["swu"])
    W["wdq"], W["wdqT"], W["swd"] = fp8bs.empty_quant_128x128(2048, 7168, batch=G)
    fp8bs.fp8_quant_128x128(d["W_down"].cuda(), W["wdq"], W["wdqT"], W["swd"])
    cap = fp8bs.fp8bs_padded_tokens_max(M, G)
    offd = _dev(off1)
    og = _moe_outputs(G, cap)
    _moe_pass(og, offd, inp, W, True)         # warm-up (first-use set-up happens outside capture)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _moe_pass(og, offd, inp, W, True)
    for routing, off in ((1, off1), (2, off2)):
        offd.copy_(torch.from_numpy(off.astype(np.int32)))
        for t in og.values():
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert fp8bs.fp8bs_last_device_status(reset=True) == 0
        mp = fp8bs.fp8bs_padded_tokens(M, off)
        oh = _moe_outputs(G, mp)
        _moe_pass(oh, off, inp, W)
        torch.cuda.synchronize()
        for k in og:
            g, h = _raw(og[k]), _raw(oh[k])
            if k in ("aT", "dyT"):
                g = g[:, :mp]
            elif k in ("saT", "sdyT"):
                g = g[:mp // 128]
            elif k in ("sx", "sa", "sdy"):
                g, h = g[:, :M], h[:, :M]
            assert np.array_equal(g, h), (routing, k)
        counts = np.diff(off)
        nonempty = [e for e in range(G) if counts[e] > 0]
        experts = sorted({nonempty[0], nonempty[-1], int(np.argmax(counts))})
        _check_moe_against_oracle(og, d, off, d, experts, seed=routing)
        del oh
