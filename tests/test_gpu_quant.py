"""GPU parity of the quantizers (S1 1x128, S2 128x128, S3 128x1 transposed)
against the CPU oracle: payload bytes and fp32 scale bits must be identical.
Inputs are seeded (workloads.py); sizes span several tiles and ragged tails,
plus the full-size tensors of the dense, backward and bandwidth workloads."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs
import oracle
import workloads as wl
from parity import np_, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fp8bs.build()
    fp8bs.lib()
    torch.cuda.init()
    yield
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def _special_inputs(R, C, seed):
    """N(0,1) with 1% outliers, an all-zero tile, a tile of tiny negatives
    and exact -0 inputs (-0 results), a tile whose absmax is negative (with
    a +0 and a -0 input), a tile with amax 448
    (scale 1) holding exact E4M3 midpoints (ties to even), and a tile of
    values around 1e-20 (a scale below 2^-60, where the kernels divide
    exactly instead of using the reciprocal path)."""
    x = wl.with_outliers((R, C), fraction=0.01, seed=seed)
    w = min(C, 128)
    if R > 0:
        x[0, :w] = 0.0
    if R > 1:
        x[1, :w] = -1e-30
        x[1, 2:w:3] = -0.0
        x[1, 0] = 1.0
    if R > 2:
        x[2, :w] = torch.linspace(-300.0, 2.0, w).to(torch.bfloat16)
        if w > 6:
            x[2, 5] = 0.0
            x[2, 6] = -0.0
    if R > 3:
        t = oracle.e4m3_table()
        fin = t[:0x7E].astype(np.float64)
        mids = ((fin[:-1] + fin[1:]) / 2)
        mids = mids[(mids > 0.01) & (mids < 448)]
        bf = torch.tensor(mids, dtype=torch.float32).to(torch.bfloat16)
        exact = bf.float().numpy() == mids.astype(np.float32)
        vals = bf[torch.from_numpy(exact)][: w - 1]
        row = torch.zeros(w, dtype=torch.bfloat16)
        row[0] = 448.0
        row[1:1 + vals.numel()] = vals * torch.where(torch.arange(vals.numel()) % 2 == 0, 1.0, -1.0).to(torch.bfloat16)
        x[3, :w] = row
    if R > 4:
        x[4, :w] = (wl.normal((w,), seed=seed + 99).float() * 1e-20).to(torch.bfloat16)
    return x


def _gpu_quant_1x128(x):
    xd = x.cuda()
    q, sc = fp8bs.empty_quant_1x128(*x.shape)
    fp8bs.fp8_quant_1x128(xd, q, sc)
    torch.cuda.synchronize()
    return np_(q), np_(sc)


def _check_1x128(x):
    R, C = x.shape
    q, sc = _gpu_quant_1x128(x)
    oq, osc = oracle.quant_1x128(u16(x))
    assert np.array_equal(q, oq)
    assert np.array_equal(sc[:, :R].view(np.uint32), osc[:, :R].view(np.uint32))


@pytest.mark.parametrize("R,C", [(1, 128), (4, 16), (37, 640), (129, 304), (300, 16), (64, 1024)])
def test_quant_1x128_small(R, C):
    _check_1x128(_special_inputs(R, C, seed=R * 7 + C))


def test_quant_1x128_negative_zero_and_ties():
    x = _special_inputs(8, 256, seed=3)
    q, sc = _gpu_quant_1x128(x)
    assert np.all(q[1, 1:128] == 0x80)                 # tiny negatives -> -0
    assert q[1, 0] == 0x7E
    assert sc[0, 0] == 1.0 and np.all(q[0, :128] == 0) # all-zero tile
    assert sc[0, 3] == 1.0                             # amax 448 -> scale 1
    oq, _ = oracle.quant_1x128(u16(x))
    assert np.array_equal(q[3], oq[3])                 # exact midpoints: ties to even


def test_quant_1x128_dense_activation_full():
    x = wl.dense(K=7168, M=4096, N=128)["X"]
    _check_1x128(x)


def test_quant_1x128_backward_grad_full():
    _check_1x128(wl.normal((4096, 2048), std=wl.DY_STD, seed=2))


@pytest.mark.slow
def test_quant_1x128_stream_16k_full():
    _check_1x128(wl.quant_stream()["X"])


def _gpu_quant_128x128(w):
    wd = w.cuda()
    batch = w.shape[0] if w.dim() == 3 else None
    q, qT, sc = fp8bs.empty_quant_128x128(w.shape[-2], w.shape[-1], batch=batch)
    fp8bs.fp8_quant_128x128(wd, q, qT, sc)
    torch.cuda.synchronize()
    return np_(q), np_(qT), np_(sc)


@pytest.mark.parametrize("R,C", [(128, 128), (512, 256), (144, 400), (16, 16), (384, 1040)])
def test_quant_128x128_small(R, C):
    w = _special_inputs(R, C, seed=R + C)
    q, qT, sc = _gpu_quant_128x128(w)
    oq, osc = oracle.quant_128x128(u16(w))
    assert np.array_equal(q, oq)
    assert np.array_equal(sc.view(np.uint32), osc.view(np.uint32))
    assert np.array_equal(qT, oq.T)


def test_quant_128x128_batched_experts():
    w = wl.normal((3, 256, 384), std=wl.W_STD, seed=5)
    q, qT, sc = _gpu_quant_128x128(w)
    for e in range(3):
        oq, osc = oracle.quant_128x128(u16(w[e]))
        assert np.array_equal(q[e], oq)
        assert np.array_equal(qT[e], oq.T)
        assert np.array_equal(sc[e], osc)


@pytest.mark.parametrize("B,R,C", [(3, 144, 400), (2, 16, 16), (4, 272, 144)])
def test_quant_128x128_batched_ragged(B, R, C):
    """Batched weights whose rows are not a multiple of 128: a block at an
    expert's ragged edge must not read the next expert's rows (they count as
    zeros), and every expert's codes, transposed copy and scales equal the
    oracle's cast of that expert alone."""
    w = torch.stack([_special_inputs(R, C, seed=100 * b + R + C) for b in range(B)])
    q, qT, sc = _gpu_quant_128x128(w)
    for e in range(B):
        oq, osc = oracle.quant_128x128(u16(w[e]))
        assert np.array_equal(q[e], oq), f"expert {e}"
        assert np.array_equal(qT[e], oq.T), f"expert {e} transposed"
        assert np.array_equal(sc[e].view(np.uint32), osc.view(np.uint32)), f"expert {e} scales"


@pytest.mark.parametrize("shape", [(7168, 2048), (3, 208, 384)])
def test_quant_128x128_without_transpose(shape):
    """The weight cast without its transposed copy (qT NULL: Fprop reading
    the codes as stored): codes and scales equal the oracle's, for the dense
    weight and for batched experts with a ragged edge, under round to nearest
    and under stochastic rounding."""
    w = (wl.dense(M=128)["W"] if len(shape) == 2 else
         torch.stack([_special_inputs(shape[1], shape[2], seed=7 + b) for b in range(shape[0])]))
    R, C = w.shape[-2:]
    batch = w.shape[0] if w.dim() == 3 else None
    wd = w.cuda()
    q, _, sc = fp8bs.empty_quant_128x128(R, C, batch=batch, with_transpose=False)
    fp8bs.fp8_quant_128x128(wd, q, None, sc)
    q2, qT2, sc2 = fp8bs.empty_quant_128x128(R, C, batch=batch)
    fp8bs.fp8_quant_128x128_sr(wd, q2, qT2, sc2, seed=11, salt=2)
    qs, _, scs = fp8bs.empty_quant_128x128(R, C, batch=batch, with_transpose=False)
    fp8bs.fp8_quant_128x128_sr(wd, qs, None, scs, seed=11, salt=2)
    torch.cuda.synchronize()
    assert torch.equal(qs, q2) and torch.equal(scs, sc2)   # SR codes do not depend on the transpose
    ws = [w] if batch is None else list(w)
    qn, scn = np_(q).reshape(-1, R, C), np_(sc).reshape(len(ws), -1)
    for e, we in enumerate(ws):
        oq, osc = oracle.quant_128x128(u16(we))
        assert np.array_equal(qn[e], oq), f"entry {e}"
        assert np.array_equal(scn[e].view(np.uint32), osc.reshape(-1).view(np.uint32)), f"entry {e} scales"


def test_quant_128x128_dense_weight_full():
    w = wl.dense(M=128)["W"]
    q, qT, sc = _gpu_quant_128x128(w)
    oq, osc = oracle.quant_128x128(u16(w))
    assert np.array_equal(q, oq)
    assert np.array_equal(sc.view(np.uint32), osc.view(np.uint32))
    assert np.array_equal(qT, oq.T)


def _gpu_requant(src, src_scales=None, offsets=None):
    qT, scT = fp8bs.empty_requant_128x1_T(src.shape[0], src.shape[1], offsets)
    fp8bs.fp8_requant_128x1_T(src, src_scales, qT, scT, offsets=offsets)
    torch.cuda.synchronize()
    return np_(qT), np_(scT)


@pytest.mark.parametrize("M,C,counts", [
    (128, 128, None), (300, 256, None), (1, 16, None), (257, 400, None),
    (400, 128, [0, 129, 1, 0, 270]), (131, 144, [131]), (260, 256, [0, 0, 260, 0]),
])
def test_requant_bf16_source(M, C, counts):
    x = _special_inputs(M, C, seed=M + 3 * C)
    off = None if counts is None else wl.offsets_from_counts(counts)
    qT, scT = _gpu_requant(x.cuda(), None, off)
    oqT, oscT = oracle.requant_128x1_T(u16(x), offsets=off)
    assert np.array_equal(qT, oqT)
    assert np.array_equal(scT.view(np.uint32), oscT.view(np.uint32))


@pytest.mark.parametrize("M,C,counts", [
    (128, 128, None), (300, 256, None), (257, 400, None), (400, 128, [0, 129, 1, 0, 270]),
])
def test_requant_e4m3_stash_source(M, C, counts):
    x = _special_inputs(M, C, seed=M + 5 * C)
    xq, sx = fp8bs.empty_quant_1x128(M, C)
    fp8bs.fp8_quant_1x128(x.cuda(), xq, sx)
    off = None if counts is None else wl.offsets_from_counts(counts)
    qT, scT = _gpu_requant(xq, sx, off)
    oq, osc = oracle.quant_1x128(u16(x))
    oqT, oscT = oracle.requant_128x1_T(oq, osc, offsets=off)
    assert np.array_equal(qT, oqT)
    assert np.array_equal(scT.view(np.uint32), oscT.view(np.uint32))


def test_requant_backward_full():
    """The backward workload's two requants: X from its E4M3 stash, dY from BF16."""
    d = wl.backward()
    x, dy = d["X"], d["dY"]
    xq, sx = fp8bs.empty_quant_1x128(*x.shape)
    fp8bs.fp8_quant_1x128(x.cuda(), xq, sx)
    qT, scT = _gpu_requant(xq, sx)
    oq, osc = oracle.quant_1x128(u16(x))
    oqT, oscT = oracle.requant_128x1_T(oq, osc)
    assert np.array_equal(qT, oqT) and np.array_equal(scT, oscT)
    qT, scT = _gpu_requant(dy.cuda())
    oqT, oscT = oracle.requant_128x1_T(u16(dy))
    assert np.array_equal(qT, oqT) and np.array_equal(scT, oscT)


def test_requant_moe_grouped_full_tokens():
    d = wl.moe(with_weights=False)
    dy = d["dY"]
    qT, scT = _gpu_requant(dy.cuda(), None, d["offsets"])
    oqT, oscT = oracle.requant_128x1_T(u16(dy), offsets=d["offsets"])
    assert np.array_equal(qT, oqT) and np.array_equal(scT, oscT)


def test_quantizers_are_deterministic():
    x = _special_inputs(300, 512, seed=9)
    a = _gpu_quant_1x128(x)
    b = _gpu_quant_1x128(x)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def _gpu_dual(x_dev, offsets=None):
    R, C = x_dev.shape
    q, sc = fp8bs.empty_quant_1x128(R, C)
    qT, scT = fp8bs.empty_requant_128x1_T(R, C, offsets)
    fp8bs.fp8_quant_dual(x_dev, q, sc, qT, scT, offsets=offsets)
    torch.cuda.synchronize()
    return np_(q), np_(sc), np_(qT), np_(scT)


def _check_dual(x, offsets=None):
    R, C = x.shape
    q, sc, qT, scT = _gpu_dual(x.cuda(), offsets)
    oq, osc = oracle.quant_1x128(u16(x))
    assert np.array_equal(q, oq)
    assert np.array_equal(sc[:, :R].view(np.uint32), osc[:, :R].view(np.uint32))
    oqT, oscT = oracle.requant_128x1_T(u16(x), offsets=offsets)
    assert np.array_equal(qT, oqT)
    assert np.array_equal(scT.view(np.uint32), oscT.view(np.uint32))


@pytest.mark.parametrize("M,C,counts", [
    (128, 128, None), (300, 256, None), (1, 16, None), (257, 400, None), (129, 2048, None),
    (400, 128, [0, 129, 1, 0, 270]), (131, 144, [131]), (260, 256, [0, 0, 260, 0]),
])
def test_quant_dual_matches_both_casts(M, C, counts):
    """One read of BF16 dY gives the 1x128 cast and the 128x1 transposed cast,
    byte-identical to the oracle's two quantizations (special tiles included:
    zeros, -0 and tiny negatives, exact E4M3 midpoints, tiny scales)."""
    x = _special_inputs(M, C, seed=M + 7 * C)
    _check_dual(x, None if counts is None else wl.offsets_from_counts(counts))


def test_quant_dual_backward_grad_full():
    _check_dual(wl.backward()["dY"])


def test_quant_dual_moe_grouped_full():
    d = wl.moe(with_weights=False)
    _check_dual(d["dY"], d["offsets"])


def _gpu_dual_stash(x_dev, offsets=None, **r):
    R, C = x_dev.shape
    q, sc = fp8bs.empty_quant_1x128(R, C)
    qT, scT = fp8bs.empty_requant_128x1_T(R, C, offsets)
    fp8bs.fp8_quant_dual_stash(x_dev, q, sc, qT, scT, offsets=offsets, **r)
    torch.cuda.synchronize()
    return np_(q), np_(sc), np_(qT), np_(scT)


def _check_dual_stash(x, offsets=None):
    R, C = x.shape
    q, sc, qT, scT = _gpu_dual_stash(x.cuda(), offsets)
    oq, osc = oracle.quant_1x128(u16(x))
    assert np.array_equal(q, oq)
    assert np.array_equal(sc[:, :R].view(np.uint32), osc[:, :R].view(np.uint32))
    oqT, oscT = oracle.requant_128x1_T(oq, osc, offsets=offsets)
    assert np.array_equal(qT, oqT)
    assert np.array_equal(scT.view(np.uint32), oscT.view(np.uint32))


@pytest.mark.parametrize("M,C,counts", [
    (128, 128, None), (300, 256, None), (1, 16, None), (257, 400, None), (129, 2048, None),
    (400, 128, [0, 129, 1, 0, 270]), (131, 144, [131]), (260, 256, [0, 0, 260, 0]),
])
def test_quant_dual_stash_matches_cast_then_requant(M, C, counts):
    """One read of BF16 X gives its 1x128 cast and the 128x1 transposed
    requant of that E4M3 stash, byte-identical to the oracle's cast followed
    by its requant of the stash (ragged token tiles and groups included)."""
    x = _special_inputs(M, C, seed=M + 11 * C)
    _check_dual_stash(x, None if counts is None else wl.offsets_from_counts(counts))


def test_quant_dual_stash_equals_two_calls_full():
    """At the dense workload's X (4096 x 7168): the fused call and the two
    separate library calls (cast, then requant of the stash) agree byte for
    byte; the oracle checks a sample of token tiles."""
    x = wl.backward()["X"]
    xd = x.cuda()
    q, sc, qT, scT = _gpu_dual_stash(xd)
    q2, sc2 = fp8bs.empty_quant_1x128(*x.shape)
    fp8bs.fp8_quant_1x128(xd, q2, sc2)
    qT2, scT2 = fp8bs.empty_requant_128x1_T(*x.shape)
    fp8bs.fp8_requant_128x1_T(q2, sc2, qT2, scT2)
    torch.cuda.synchronize()
    assert np.array_equal(q, np_(q2)) and np.array_equal(sc, np_(sc2))
    assert np.array_equal(qT, np_(qT2)) and np.array_equal(scT.view(np.uint32), np_(scT2).view(np.uint32))
    rows = slice(1280, 1536)                       # two token tiles
    oq, osc = oracle.quant_1x128(u16(x[rows]))
    oqT, oscT = oracle.requant_128x1_T(oq, osc)
    assert np.array_equal(qT[:, rows], oqT) and np.array_equal(scT[10:12], oscT)


def test_quant_dual_stash_moe_grouped_full():
    d = wl.moe(with_weights=False)
    _check_dual_stash(d["dY"][:, :1024].contiguous(), d["offsets"])


RULES = [
    dict(rule=fp8bs.SCALE_UE8M0),
    dict(amax_floor=1e-4),
    dict(scale_floor=2.0 ** -33),
    dict(rule=fp8bs.SCALE_UE8M0, scale_floor=2.0 ** -33),
    dict(rule=fp8bs.SCALE_UE8M0, amax_floor=1e-4),
]


def _oracle_rule(r):
    return oracle.scale_rule(ue8m0=r.get("rule", 0) == fp8bs.SCALE_UE8M0,
                             amax_floor=r.get("amax_floor", 0.0), scale_floor=r.get("scale_floor", 0.0))


@pytest.mark.parametrize("r", RULES)
def test_scale_rules_all_quantizers(r):
    """Scale rules (UE8M0 scales, amax and scale floors) on every
    quantizer, byte- and bit-exact against the oracle under the same rule;
    the inputs include an all-zero tile, where the floors decide the scale."""
    M, C = 300, 384
    x = _special_inputs(M, C, seed=31)
    xd = x.cuda()
    q, sc = fp8bs.empty_quant_1x128(M, C)
    fp8bs.fp8_quant_1x128(xd, q, sc, **r)
    w = _special_inputs(384, 256, seed=32)
    wq, wqT, sw = fp8bs.empty_quant_128x128(384, 256)
    fp8bs.fp8_quant_128x128(w.cuda(), wq, wqT, sw, **r)
    off = wl.offsets_from_counts([0, 129, 1, 0, 170])
    qT, scT = fp8bs.empty_requant_128x1_T(M, C, off)
    fp8bs.fp8_requant_128x1_T(xd, None, qT, scT, offsets=off, **r)
    xq0, sx0 = fp8bs.empty_quant_1x128(M, C)
    fp8bs.fp8_quant_1x128(xd, xq0, sx0)                     # default-rule stash
    qTq, scTq = fp8bs.empty_requant_128x1_T(M, C)
    fp8bs.fp8_requant_128x1_T(xq0, sx0, qTq, scTq, **r)
    dq, dsc = fp8bs.empty_quant_1x128(M, C)
    dqT, dscT = fp8bs.empty_requant_128x1_T(M, C, off)
    fp8bs.fp8_quant_dual(xd, dq, dsc, dqT, dscT, offsets=off, **r)
    sq, ssc, sqT, sscT = _gpu_dual_stash(xd, off, **r)
    torch.cuda.synchronize()

    oxq0, osx0 = oracle.quant_1x128(u16(x))
    with _oracle_rule(r):
        oq, osc = oracle.quant_1x128(u16(x))
        owq, osw = oracle.quant_128x128(u16(w))
        oqT, oscT = oracle.requant_128x1_T(u16(x), offsets=off)
        oqTq, oscTq = oracle.requant_128x1_T(oxq0, osx0)
        oqTs, oscTs = oracle.requant_128x1_T(oq, osc, offsets=off)
    bits = lambda a: np.ascontiguousarray(a).view(np.uint32)
    assert np.array_equal(np_(q), oq) and np.array_equal(bits(np_(sc)[:, :M]), bits(osc[:, :M]))
    assert np.array_equal(np_(wq), owq) and np.array_equal(bits(np_(sw)), bits(osw))
    assert np.array_equal(np_(wqT), owq.T)
    assert np.array_equal(np_(qT), oqT) and np.array_equal(bits(np_(scT)), bits(oscT))
    assert np.array_equal(np_(qTq), oqTq) and np.array_equal(bits(np_(scTq)), bits(oscTq))
    assert np.array_equal(np_(dq), oq) and np.array_equal(bits(np_(dsc)[:, :M]), bits(osc[:, :M]))
    assert np.array_equal(np_(dqT), oqT) and np.array_equal(bits(np_(dscT)), bits(oscT))
    assert np.array_equal(sq, oq) and np.array_equal(bits(ssc[:, :M]), bits(osc[:, :M]))
    assert np.array_equal(sqT, oqTs) and np.array_equal(bits(sscT), bits(oscTs))
    if r.get("rule") == fp8bs.SCALE_UE8M0:
        mant, _ = np.frexp(np_(sc)[:, :M])
        assert np.all(mant == 0.5)


def test_scale_rule_rejects_bad_options():
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device="cuda")
    q, sc = fp8bs.empty_quant_1x128(4, 128)
    for bad in (dict(rule=7), dict(amax_floor=-1.0), dict(scale_floor=float("nan"))):
        with pytest.raises(fp8bs.Fp8bsError):
            fp8bs.fp8_quant_1x128(x, q, sc, **bad)


@pytest.mark.parametrize("R,C,seed,salt", [(300, 384, 0, 0), (129, 2048, 2 ** 40 + 17, 3), (1, 16, 7, 0xFFFFFFFF)])
def test_sr_quant_1x128_matches_oracle(R, C, seed, salt):
    """Stochastic rounding under (seed, salt), byte- and bit-exact
    against the oracle's independent Philox4x32-10 and rounding rule."""
    x = _special_inputs(R, C, seed=R + C + 5)
    q, sc = fp8bs.empty_quant_1x128(R, C)
    fp8bs.fp8_quant_1x128_sr(x.cuda(), q, sc, seed=seed, salt=salt)
    torch.cuda.synchronize()
    oq, osc = oracle.quant_1x128_sr(u16(x), seed=seed, salt=salt)
    assert np.array_equal(np_(q), oq)
    assert np.array_equal(np_(sc)[:, :R].view(np.uint32), osc[:, :R].view(np.uint32))


def test_sr_quant_128x128_batched_matches_oracle():
    w = wl.normal((3, 256, 384), std=wl.W_STD, seed=41)
    w[1, :128, :128] = 0.0
    q, qT, sc = fp8bs.empty_quant_128x128(256, 384, batch=3)
    fp8bs.fp8_quant_128x128_sr(w.cuda(), q, qT, sc, seed=99, salt=5)
    torch.cuda.synchronize()
    for e in range(3):
        oq, osc = oracle.quant_128x128_sr(u16(w[e]), seed=99, salt=5, idx_base=e * 256 * 384)
        assert np.array_equal(np_(q)[e], oq)
        assert np.array_equal(np_(qT)[e], oq.T)
        assert np.array_equal(np_(sc)[e].view(np.uint32), osc.view(np.uint32))


@pytest.mark.parametrize("M,C,counts,seed,salt", [
    (128, 128, None, 0, 0), (300, 256, None, 2 ** 40 + 17, 3), (257, 400, None, 7, 0xFFFFFFFF),
    (400, 128, [0, 129, 1, 0, 270], 11, 5),
])
def test_sr_requant_both_sources_match_oracle(M, C, counts, seed, salt):
    """Stochastic rounding on the transposed cast from BF16 and from
    an E4M3 stash, byte- and bit-exact against the oracle (source element
    (r, c) takes word r * C + c; ragged token tiles and groups included)."""
    x = _special_inputs(M, C, seed=M + 13 * C)
    off = None if counts is None else wl.offsets_from_counts(counts)
    xd = x.cuda()
    qT, scT = fp8bs.empty_requant_128x1_T(M, C, off)
    fp8bs.fp8_requant_128x1_T_sr(xd, None, qT, scT, seed=seed, salt=salt, offsets=off)
    xq, sx = fp8bs.empty_quant_1x128(M, C)
    fp8bs.fp8_quant_1x128(xd, xq, sx)
    qTq, scTq = fp8bs.empty_requant_128x1_T(M, C, off)
    fp8bs.fp8_requant_128x1_T_sr(xq, sx, qTq, scTq, seed=seed, salt=salt, offsets=off)
    torch.cuda.synchronize()
    oqT, oscT = oracle.requant_128x1_T_sr(u16(x), offsets=off, seed=seed, salt=salt)
    assert np.array_equal(np_(qT), oqT)
    assert np.array_equal(np_(scT).view(np.uint32), oscT.view(np.uint32))
    oq, osc = oracle.quant_1x128(u16(x))
    oqTq, oscTq = oracle.requant_128x1_T_sr(oq, osc, offsets=off, seed=seed, salt=salt)
    assert np.array_equal(np_(qTq), oqTq)
    assert np.array_equal(np_(scTq).view(np.uint32), oscTq.view(np.uint32))


@pytest.mark.parametrize("stash", [False, True])
@pytest.mark.parametrize("M,C,counts", [(300, 256, None), (400, 128, [0, 129, 1, 0, 270])])
def test_sr_dual_and_stash_match_oracle(stash, M, C, counts):
    """The SR dual and stash casts: the 1x128 part is the oracle's SR cast
    under (seed, salt), the transposed part the oracle's SR requant under
    (seed, salt + 1) of the BF16 values (dual) or of that SR stash (stash)."""
    seed, salt = 77, 9
    x = _special_inputs(M, C, seed=M + 17 * C)
    off = None if counts is None else wl.offsets_from_counts(counts)
    q, sc = fp8bs.empty_quant_1x128(M, C)
    qT, scT = fp8bs.empty_requant_128x1_T(M, C, off)
    fn = fp8bs.fp8_quant_dual_stash_sr if stash else fp8bs.fp8_quant_dual_sr
    fn(x.cuda(), q, sc, qT, scT, seed=seed, salt=salt, offsets=off)
    torch.cuda.synchronize()
    oq, osc = oracle.quant_1x128_sr(u16(x), seed=seed, salt=salt)
    assert np.array_equal(np_(q), oq)
    assert np.array_equal(np_(sc)[:, :M].view(np.uint32), osc[:, :M].view(np.uint32))
    src = (oq, osc) if stash else (u16(x), None)
    oqT, oscT = oracle.requant_128x1_T_sr(src[0], src[1], offsets=off, seed=seed, salt=salt + 1)
    assert np.array_equal(np_(qT), oqT)
    assert np.array_equal(np_(scT).view(np.uint32), oscT.view(np.uint32))


def test_sr_stash_full_dense_x_sampled():
    """The fused SR cast of the dense X (4096 x 7168) against the two separate
    SR library calls in full and the oracle on the first two token tiles."""
    x = wl.backward()["X"]
    xd = x.cuda()
    M, C = x.shape
    q, sc = fp8bs.empty_quant_1x128(M, C)
    qT, scT = fp8bs.empty_requant_128x1_T(M, C)
    fp8bs.fp8_quant_dual_stash_sr(xd, q, sc, qT, scT, seed=5, salt=6)
    q2, sc2 = fp8bs.empty_quant_1x128(M, C)
    fp8bs.fp8_quant_1x128_sr(xd, q2, sc2, seed=5, salt=6)
    qT2, scT2 = fp8bs.empty_requant_128x1_T(M, C)
    fp8bs.fp8_requant_128x1_T_sr(q2, sc2, qT2, scT2, seed=5, salt=7)
    torch.cuda.synchronize()
    assert np.array_equal(np_(q), np_(q2)) and np.array_equal(np_(qT), np_(qT2))
    assert np.array_equal(np_(scT).view(np.uint32), np_(scT2).view(np.uint32))
    rows = slice(0, 256)                  # the oracle's element indices start at row 0
    oq, osc = oracle.quant_1x128_sr(u16(x)[rows], seed=5, salt=6)
    assert np.array_equal(np_(q)[rows], oq)


def test_sr_full_size_and_statistics():
    """The dense activation in full under SR equals the oracle, differs from
    round-to-nearest on a sizeable fraction of elements, and another salt
    gives another draw."""
    x = wl.dense(K=7168, M=1024, N=128)["X"]
    R, C = x.shape
    q, sc = fp8bs.empty_quant_1x128(R, C)
    fp8bs.fp8_quant_1x128_sr(x.cuda(), q, sc, seed=2024, salt=1)
    q2, _ = fp8bs.empty_quant_1x128(R, C)
    fp8bs.fp8_quant_1x128_sr(x.cuda(), q2, sc, seed=2024, salt=2)
    torch.cuda.synchronize()
    oq, _ = oracle.quant_1x128_sr(u16(x), seed=2024, salt=1)
    assert np.array_equal(np_(q), oq)
    rn, _ = oracle.quant_1x128(u16(x))
    assert 0.2 < np.mean(np_(q) != rn) < 0.6
    assert np.mean(np_(q) != np_(q2)) > 0.2
