"""GPU parity of the grouped (MoE expert) MX path, hardware block scaling
with power-of-two scales: fp8_pack_ue8m0_grouped byte for byte against the oracle's packing of
each group's 1x128 power-of-two scales placed in the groups' tile layout, and
fp8_mx_gemm_grouped (Fprop, Dgrad, Wgrad on the tensor core's block scaling)
per expert against the oracle's promoted GEMMs of the same UE8M0-rule codes
and scales, within |d| <= 2e-3 * sum_k |a_k b_k| + 1e-6 (plus one BF16 ulp for
BF16 outputs), including empty experts, with host and with device offsets.
The oracle's codes and scales come from its own casts under the UE8M0 rule;
the GPU casts are checked equal to them byte for byte first."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs
import oracle
import workloads as wl
from parity import assert_gemm_close, bf16_values, np_, u16
from test_gpu_mx import atoms_to_rows

pytestmark = pytest.mark.gpu

UE8M0 = fp8bs.ScaleOpts(fp8bs.SCALE_UE8M0, 0.0, 0.0)
COUNTS = [[0, 129, 1, 0, 270], [300, 0], [128, 128]]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fp8bs.build()
    fp8bs.lib()
    torch.cuda.init()
    yield
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def _offs(off, dev):
    return torch.tensor(np.asarray(off, np.int32), dtype=torch.int32, device="cuda") if dev else off


def _tpad(M, off, dev):
    return fp8bs.fp8bs_padded_tokens_max(M, len(off) - 1) if dev else fp8bs.fp8bs_padded_tokens(M, off)


def _cast_rows(x):
    """UE8M0-rule 1x128 cast on the GPU, checked against the oracle's."""
    q, s = fp8bs.empty_quant_1x128(*x.shape)
    fp8bs.fp8_quant_1x128_opts(x.cuda(), q, s, UE8M0)
    with oracle.scale_rule(ue8m0=True):
        oq, osc = oracle.quant_1x128(u16(x))
    torch.cuda.synchronize()
    R = x.shape[0]
    assert np.array_equal(np_(q), oq) and np.array_equal(np_(s)[:, :R], osc[:, :R])
    return q, s, oq, osc


def _pack_grouped(s, M, K, off, dev):
    atoms = torch.full((fp8bs.fp8bs_mx_scale_bytes(_tpad(M, off, dev), K),), 0xEE, dtype=torch.uint8,
                       device="cuda")
    fp8bs.fp8_pack_ue8m0_grouped(s, M, K, _offs(off, dev), atoms)
    return atoms


def _dec_rows(q, s):
    t = oracle.e4m3_table().astype(np.float64)
    return t[q] * np.repeat(s.T.astype(np.float64), 128, axis=1)


def _dec_blocks(q, s):
    t = oracle.e4m3_table().astype(np.float64)
    return t[q] * np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)


@pytest.mark.parametrize("counts", COUNTS)
@pytest.mark.parametrize("dev", [False, True])
def test_pack_ue8m0_grouped_matches_oracle(counts, dev):
    off = wl.offsets_from_counts(counts)
    M, K = int(off[-1]), 384
    x = wl.with_outliers((M, K), fraction=0.01, seed=3 + len(counts))
    q, s, oq, osc = _cast_rows(x)
    atoms = _pack_grouped(s, M, K, off, dev)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    got = np_(atoms)
    per_tile = (K // 128) * 512
    t = 0
    for e in range(len(counts)):
        r0, r1 = int(off[e]), int(off[e + 1])
        n = r1 - r0
        if n == 0:
            continue
        sc = np.ascontiguousarray(osc[:, r0:r1])                  # [K/128 x n]
        ref, bad = oracle.pack_ue8m0(sc, n, K, 1, 1, n)            # exponent bytes [n x K/32]
        assert bad == 0
        tiles = -(-n // 128)
        rows = atoms_to_rows(got[t * per_tile:(t + tiles) * per_tile], tiles * 128, K)
        assert np.array_equal(rows[:n], ref), f"group {e}"
        assert np.all(rows[n:] == 127), f"group {e} padding rows"
        t += tiles
    assert np.all(got[t * per_tile:] == 0xEE)                      # nothing past the groups' tiles


@pytest.mark.parametrize("counts", COUNTS)
@pytest.mark.parametrize("dev", [False, True])
def test_grouped_mx_fprop_dgrad(counts, dev):
    off = wl.offsets_from_counts(counts)
    G, M = len(counts), int(off[-1])
    K, N = 256, 512            # Fprop: contraction K, width N; Dgrad: contraction N, width K
    x = wl.with_outliers((M, K), fraction=0.01, seed=10 + G)
    dy = wl.normal((M, N), std=wl.DY_STD, seed=11 + G)
    w = wl.normal((G, K, N), std=wl.W_STD, seed=12 + G)
    xq, sx, oxq, osx = _cast_rows(x)
    dyq, sdy, odyq, osdy = _cast_rows(dy)
    wq, wqT, sw = fp8bs.empty_quant_128x128(K, N, batch=G)
    awT, aw = fp8bs.empty_mx_atoms(N, K, batch=G), fp8bs.empty_mx_atoms(K, N, batch=G)
    fp8bs.fp8_quant_128x128_packed(w.cuda(), wq, wqT, sw, awT, aw)
    ax = _pack_grouped(sx, M, K, off, dev)
    ady = _pack_grouped(sdy, M, N, off, dev)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    dx = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_kn = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_mx_gemm_grouped(fp8bs.OP_FPROP, _offs(off, dev), xq, ax, wqT, awT, y, N, K)
    fp8bs.fp8_mx_gemm_grouped(fp8bs.OP_DGRAD, _offs(off, dev), dyq, ady, wq, aw, dx, N, K)
    # Fprop on the experts' codes as stored ([G x K x N], read MN-major)
    fp8bs.fp8_mx_gemm_grouped(fp8bs.OP_FPROP_WKN, _offs(off, dev), xq, ax, wq, awT, y_kn, N, K)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    assert torch.equal(y_kn.view(torch.int16), y.view(torch.int16))
    y, dx = bf16_values(y), bf16_values(dx)
    for e in range(G):
        r0, r1 = int(off[e]), int(off[e + 1])
        with oracle.scale_rule(ue8m0=True):
            owq, osw = oracle.quant_128x128(u16(w[e]))
        assert np.array_equal(np_(wq[e]), owq) and np.array_equal(np_(sw[e]), osw)
        if r1 == r0:
            continue
        oxe, osxe = oxq[r0:r1], np.ascontiguousarray(osx[:, r0:r1])
        ode, osde = odyq[r0:r1], np.ascontiguousarray(osdy[:, r0:r1])
        wa = np.abs(_dec_blocks(owq, osw))
        assert_gemm_close(y[r0:r1], oracle.fprop(oxe, osxe, owq, osw), np.abs(_dec_rows(oxe, osxe)) @ wa, True,
                          f"grouped mx fprop e{e}")
        assert_gemm_close(dx[r0:r1], oracle.dgrad(ode, osde, owq, osw), np.abs(_dec_rows(ode, osde)) @ wa.T, True,
                          f"grouped mx dgrad e{e}")


@pytest.mark.parametrize("counts", [[0, 129, 1, 0, 270], [128], [0, 0]])
@pytest.mark.parametrize("dev", [False, True])
def test_grouped_mx_wgrad(counts, dev):
    off = wl.offsets_from_counts(counts)
    G, M = len(counts), int(off[-1])
    N, K = 256, 512
    dy = wl.normal((M, N), std=wl.DY_STD, seed=21 + G)
    a_ = wl.with_outliers((M, K), fraction=0.01, seed=22 + G)
    tp = _tpad(M, off, dev)
    dyT = torch.zeros((N, tp), dtype=torch.uint8, device="cuda")
    aT = torch.zeros((K, tp), dtype=torch.uint8, device="cuda")
    sdyT = torch.ones((tp // 128, N), dtype=torch.float32, device="cuda")
    saT = torch.ones((tp // 128, K), dtype=torch.float32, device="cuda")
    if M:
        fp8bs.fp8_requant_128x1_T_opts(dy.cuda(), None, dyT, sdyT, UE8M0, offsets=_offs(off, dev))
        fp8bs.fp8_requant_128x1_T_opts(a_.cuda(), None, aT, saT, UE8M0, offsets=_offs(off, dev))
    ad = fp8bs.empty_mx_atoms(N, max(tp, 128))
    aa = fp8bs.empty_mx_atoms(K, max(tp, 128))
    if tp:
        fp8bs.fp8_pack_ue8m0(sdyT, N, tp, 1, 1, N, ad)
        fp8bs.fp8_pack_ue8m0(saT, K, tp, 1, 1, K, aa)
    dw = torch.full((G, N, K), float("nan"), dtype=torch.float32, device="cuda")
    fp8bs.fp8_mx_gemm_grouped(fp8bs.OP_WGRAD, _offs(off, dev), dyT, ad, aT, aa, dw, N, K, rows=M)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    dw = np_(dw)
    with oracle.scale_rule(ue8m0=True):
        odyT, osdyT = oracle.requant_128x1_T(u16(dy), offsets=off)
        oaT, osaT = oracle.requant_128x1_T(u16(a_), offsets=off)
    mp = fp8bs.fp8bs_padded_tokens(M, off)
    assert np.array_equal(np_(dyT)[:, :mp], odyT) and np.array_equal(np_(aT)[:, :mp], oaT)
    p = 0
    for e in range(G):
        n_e = int(off[e + 1] - off[e])
        w_e = -(-n_e // 128) * 128
        if n_e == 0:
            assert np.all(dw[e] == 0.0), f"empty expert {e}"
            continue
        ref = oracle.wgrad(odyT, osdyT, oaT, osaT, t0=p, t1=p + w_e)
        t = oracle.e4m3_table().astype(np.float64)
        da = t[odyT[:, p:p + w_e]] * np.repeat(osdyT[p // 128:(p + w_e) // 128].T.astype(np.float64), 128, 1)
        xa = t[oaT[:, p:p + w_e]] * np.repeat(osaT[p // 128:(p + w_e) // 128].T.astype(np.float64), 128, 1)
        assert_gemm_close(dw[e], ref, np.abs(da) @ np.abs(xa).T, False, f"grouped mx wgrad e{e}")
        p += w_e


@pytest.mark.parametrize("bad", [[1, 129, 130, 300], [0, 200, 100, 300], [0, 100, 200, 299]])
def test_grouped_mx_invalid_device_offsets_record_error_and_write_nothing(bad):
    """off[0] != 0, a decrease, a total other than rows, read by the grouped
    packing and the grouped MX GEMM when they run: FP8BS_ERR_DEVICE in the
    status word, nothing written, and the same calls with valid offsets are
    then byte-identical to their host-offset form."""
    M, K, N, G = 300, 256, 512, 3      # the output width a multiple of 256
    offd = _offs(bad, True)
    x = wl.normal((M, K), seed=70)
    q, s, _, _ = _cast_rows(x)
    atoms = _pack_grouped(s, M, K, bad, True)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 7
    assert torch.all(atoms == 0xEE)
    good = wl.offsets_from_counts([100, 0, 200])
    ax = _pack_grouped(s, M, K, good, True)
    w = wl.normal((G, K, N), std=wl.W_STD, seed=71)
    wq, wqT, sw = fp8bs.empty_quant_128x128(K, N, batch=G)
    awT, aw = fp8bs.empty_mx_atoms(N, K, batch=G), fp8bs.empty_mx_atoms(K, N, batch=G)
    fp8bs.fp8_quant_128x128_packed(w.cuda(), wq, wqT, sw, awT, aw)
    y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_mx_gemm_grouped(fp8bs.OP_FPROP, offd, q, ax, wqT, awT, y, N, K)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 7
    assert torch.all(y == 3.0)
    axh = _pack_grouped(s, M, K, good, False)
    yh = torch.empty_like(y)
    fp8bs.fp8_mx_gemm_grouped(fp8bs.OP_FPROP, good, q, axh, wqT, awT, yh, N, K)
    fp8bs.fp8_mx_gemm_grouped(fp8bs.OP_FPROP, _offs(good, True), q, ax, wqT, awT, y, N, K)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    n_host = fp8bs.fp8bs_mx_scale_bytes(fp8bs.fp8bs_padded_tokens(M, good), K)
    assert torch.equal(ax[:n_host], axh)
    assert torch.equal(y.view(torch.int16), yh.view(torch.int16))


@pytest.mark.parametrize("stash", [False, True])
@pytest.mark.parametrize("dev", [False, True])
@pytest.mark.parametrize("counts", [[0, 129, 1, 0, 270], [300, 0], [5]])
def test_grouped_packed_casts_equal_cast_then_pack(counts, dev, stash):
    """The grouped dual and stash casts that write their scales' exponent
    bytes in the same pass (q's atoms in the groups' tile layout, qT's over
    the padded tokens) equal the grouped UE8M0 casts followed by
    fp8_pack_ue8m0_grouped and fp8_pack_ue8m0, byte for byte; with device
    offsets over the groups' padded tokens of the capacity layout."""
    off = wl.offsets_from_counts(counts)
    M, G, C = int(off[-1]), len(counts), 256
    x = wl.with_outliers((M, C), fraction=0.01, seed=20 + G).cuda()
    cast = fp8bs.fp8_quant_dual_stash_opts if stash else fp8bs.fp8_quant_dual_opts
    fused = fp8bs.fp8_quant_dual_stash_packed if stash else fp8bs.fp8_quant_dual_packed
    # reference: host offsets, cast then pack
    mp = fp8bs.fp8bs_padded_tokens(M, off)
    q, sc = fp8bs.empty_quant_1x128(M, C)
    qT, scT = fp8bs.empty_requant_128x1_T(M, C, off)
    cast(x, q, sc, qT, scT, UE8M0, offsets=off)
    ra = torch.full((fp8bs.fp8bs_mx_scale_bytes(mp, C),), 0xEE, dtype=torch.uint8, device="cuda")
    fp8bs.fp8_pack_ue8m0_grouped(sc, M, C, off, ra)
    rT = torch.full((fp8bs.fp8bs_mx_scale_bytes(C, mp),), 0xEE, dtype=torch.uint8, device="cuda")
    fp8bs.fp8_pack_ue8m0(scT, C, mp, 1, 1, C, rT)
    # the fused casts
    offs = _offs(off, dev)
    mpd = _tpad(M, off, dev)
    q2, sc2 = fp8bs.empty_quant_1x128(M, C)
    qT2, scT2 = fp8bs.empty_requant_128x1_T(M, C, offs)
    a2 = torch.full((fp8bs.fp8bs_mx_scale_bytes(mpd, C),), 0xEE, dtype=torch.uint8, device="cuda")
    aT2 = torch.full((fp8bs.fp8bs_mx_scale_bytes(C, mpd),), 0xEE, dtype=torch.uint8, device="cuda")
    fused(x, q2, sc2, qT2, scT2, a2, aT2, offsets=offs)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    assert torch.equal(q2, q) and torch.equal(sc2[:, :M], sc[:, :M])
    assert torch.equal(qT2[:, :mp], qT) and torch.equal(scT2[:mp // 128], scT)
    nq = (mp // 128) * (C // 128) * 512
    assert torch.equal(a2[:nq], ra[:nq])
    t, td = mp // 128, mpd // 128
    for ct in range(C // 128):
        assert torch.equal(aT2[ct * td * 512:(ct * td + t) * 512], rT[ct * t * 512:(ct + 1) * t * 512]), ct
