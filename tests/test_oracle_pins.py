"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle's own formulas retyped.

  - printed constants (tests/golden/page_constants.txt, each line cited);
  - the E4M3 table against PyTorch's float8_e4m3fn decoding (a library
    implementation of the OCP format) and against its structure;
  - the encoder against hand-worked OCP cases (tests/golden), a brute-force
    nearest search over all BF16 inputs, and PyTorch's float8 cast;
  - the quantizers against the same steps written with torch CPU ops and the
    library cast, plus invariants that hold for any input;
  - the transposed requant against closed-form identities;
  - the promoted GEMMs against fp64 matmuls of the dequantized operands
    within the fp32 rounding bound, and an exact single-block case;
  - the drift behaviour of the partial-sum page (unpromoted error grows with
    K, promoted error stays flat);
  - negative controls: a planted mistake in the oracle makes a pin fail.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            rows.append(line.split())
    return rows


def _f(s):
    return float.fromhex(s) if "p" in s else float(s)


def _torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float32).numpy()


def _torch_cast_codes(v_f32):
    t = torch.from_numpy(np.ascontiguousarray(v_f32, np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ---------------------------------------------------------------------------
# E4M3 table and encoder
# ---------------------------------------------------------------------------

def test_page_constants():
    c = {r[0]: r[1] for r in _golden("page_constants.txt")}
    t = oracle.e4m3_table()
    finite = t[~np.isnan(t)]
    assert float(c["e4m3_max"]) == 448.0
    assert finite.max() == 448.0 and t[0x7E] == 448.0 and t[0xFE] == -448.0
    pz, nz = int(c["pos_zero_byte"], 16), int(c["neg_zero_byte"], 16)
    assert t[pz] == 0.0 and not np.signbit(t[pz])
    assert t[nz] == 0.0 and np.signbit(t[nz])
    assert oracle.e4m3_encode(0.0) == pz and oracle.e4m3_encode(-0.0) == nz
    n_c = int(c["n_c"])
    assert n_c == 128
    # tile geometry: number of scales per tiling
    for (R, C) in [(1, 1), (5, 300), (128, 128), (129, 257), (300, 16)]:
        x = np.zeros((R, C), np.uint16)
        _, s1 = oracle.quant_1x128(x, sc_layout="row_major")
        assert s1.shape == (R, -(-C // n_c))
        _, s2 = oracle.quant_128x128(x)
        assert s2.shape == (-(-R // n_c), -(-C // n_c))
        _, s3 = oracle.requant_128x1_T(x)
        assert s3.shape == (-(-R // n_c), C)
    assert c["act_tile"] == "1x128" and c["weight_tile"] == "128x128" and c["wgrad_tile"] == "128x1"


def test_table_matches_torch_float8():
    ours = oracle.e4m3_table()
    ref = _torch_e4m3_values()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin].view(np.uint32), ref[fin].view(np.uint32))


def test_table_structure():
    t = oracle.e4m3_table()
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.count_nonzero(~np.isnan(t)) == 254
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)                      # monotone over positive codes
    assert np.array_equal(t[0x80:0xFF], -t[:0x7F])       # sign-magnitude
    assert t[0x01] == 2.0 ** -9 and t[0x08] == 2.0 ** -6  # smallest subnormal / normal
    assert t[0x07] == 7 * 2.0 ** -9


def test_encoder_golden_cases():
    for v, code in _golden("e4m3_rounding_cases.txt"):
        assert oracle.e4m3_encode(_f(v)) == int(code, 16), v


def test_encoder_roundtrip():
    t = oracle.e4m3_table()
    for c in range(256):
        if not np.isnan(t[c]):
            assert oracle.e4m3_encode(t[c]) == c


def _bruteforce_encode(v):
    """Nearest finite E4M3 by exhaustive search (ties to the even code),
    saturating, zero keeps the sign. Independent of the oracle's bisection."""
    t = _torch_e4m3_values().astype(np.float64)
    pos_codes = np.arange(0x7F)
    vals = t[pos_codes]
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[:, None] - vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = cand & (pos_codes[None, :] % 2 == 0)
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    pick = np.where(a >= 448.0, 0x7E, pick)
    return (pick | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def test_encoder_bruteforce_all_bf16():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = oracle.bf16_to_f32(h)
    v = v[np.isfinite(v)]
    ours = oracle.e4m3_encode_array(v)
    for chunk in range(0, v.size, 8192):
        sl = slice(chunk, chunk + 8192)
        assert np.array_equal(ours[sl], _bruteforce_encode(v[sl]))


def test_encoder_matches_torch_cast_fp32():
    g = np.random.default_rng(1)
    # random fp32 bit patterns over the E4M3 range plus midpoints
    mags = np.exp2(g.uniform(-12, np.log2(460), 400000)).astype(np.float32)
    t = _torch_e4m3_values()
    fin = t[:0x7E]
    mids = ((fin[:-1].astype(np.float64) + fin[1:]) / 2).astype(np.float32)
    v = np.concatenate([mags, -mags, mids, -mids,
                        np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    v = v[np.abs(v) < 464.0]  # torch's cast is not saturating beyond
    assert np.array_equal(oracle.e4m3_encode_array(v), _torch_cast_codes(v))


def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(2)
    v = np.concatenate([g.standard_normal(100000).astype(np.float32) * 1e3,
                        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 3.4e38], np.float32)])
    ours = oracle.f32_to_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ---------------------------------------------------------------------------
# Quantizers
# ---------------------------------------------------------------------------

def _tile_inputs(R, C, seed):
    """N(0,1) BF16 with outliers, an all-zero tile, a tile of tiny negatives,
    and a tile whose absmax element is negative."""
    x = wl.with_outliers((R, C), fraction=0.01, seed=seed)
    x[0, :128] = 0.0
    if R > 1:
        x[1, :128] = -1e-30
        x[1, 0] = 1.0
    if R > 2:
        x[2, :128] = torch.linspace(-300.0, 2.0, 128).to(torch.bfloat16)
    return wl.bits(x)


def _torch_quant_rows(v):
    """Reference steps with torch CPU ops: amax, s = amax / 448 (fp32 div),
    q = float8_e4m3fn cast of fp32(v / s)."""
    t = torch.from_numpy(v)
    amax = t.abs().amax(dim=-1, keepdim=True)
    s = torch.where(amax == 0, torch.ones_like(amax), amax / torch.tensor(448.0))
    q = (t / s).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.numpy(), s.squeeze(-1).numpy()


def test_quant_1x128_matches_torch_steps():
    R, C = 37, 128 * 5
    x = _tile_inputs(R, C, seed=3)
    q, sc = oracle.quant_1x128(x, sc_layout="row_major")
    v = oracle.bf16_to_f32(x).reshape(R, C // 128, 128)
    qr, sr = _torch_quant_rows(v)
    assert np.array_equal(q.reshape(R, C // 128, 128), qr)
    assert np.array_equal(sc.view(np.uint32), sr.view(np.uint32))
    # the tile-major layout holds the same numbers, row index contiguous
    q2, sc2 = oracle.quant_1x128(x)
    assert np.array_equal(q2, q)
    assert sc2.shape == (C // 128, 40)
    assert np.array_equal(sc2[:, :R].T, sc) and np.all(sc2[:, R:] == 0)


def test_quant_1x128_ragged_last_tile():
    R, C = 9, 128 * 2 + 48
    x = _tile_inputs(R, C, seed=4)
    q, sc = oracle.quant_1x128(x, sc_layout="row_major")
    v = oracle.bf16_to_f32(x)
    qr, sr = _torch_quant_rows(np.ascontiguousarray(v[:, 256:]))
    assert np.array_equal(q[:, 256:], qr)
    assert np.array_equal(sc[:, 2], sr)


def test_quant_128x128_matches_torch_steps():
    R, C = 256 + 40, 384
    x = _tile_inputs(R, C, seed=5)
    q, sc = oracle.quant_128x128(x)
    v = oracle.bf16_to_f32(x)
    for bi in range(sc.shape[0]):
        for bj in range(sc.shape[1]):
            blk = np.ascontiguousarray(v[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128])
            qr, sr = _torch_quant_rows(blk.reshape(1, -1))
            assert sc[bi, bj] == sr[0]
            assert np.array_equal(q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128].ravel(), qr[0])


def test_quant_invariants():
    R, C = 64, 128 * 4
    x = _tile_inputs(R, C, seed=6)
    q, sc = oracle.quant_1x128(x, sc_layout="row_major")
    t = oracle.e4m3_table()
    v = oracle.bf16_to_f32(x).reshape(R, -1, 128)
    dq = t[q].reshape(R, -1, 128)
    assert np.all(np.abs(dq) <= 448.0)
    nz = np.abs(v).max(-1) > 0
    # zero tiles: s = 1, signed zeros
    assert np.all(sc[~nz] == 1.0)
    zq = q.reshape(R, -1, 128)[~nz]
    zv = v[~nz]
    assert np.array_equal(zq, np.where(np.signbit(zv), 0x80, 0x00).astype(np.uint8))
    # the absmax element of each non-zero tile encodes to +-448
    idx = np.abs(v).argmax(-1)
    top = np.take_along_axis(dq, idx[..., None], -1)[..., 0]
    normal = sc >= np.finfo(np.float32).tiny
    assert np.all(np.abs(top[nz & normal]) == 448.0)
    # relative error of each element within half an E4M3 step (2^-4) in the normal range
    quot = v / sc[..., None]
    sel = np.abs(quot) >= 2.0 ** -6
    assert np.all(np.abs(dq[sel] - quot[sel]) <= 2.0 ** -4 * np.abs(quot[sel]))
    # signs agree (including zeros)
    assert np.array_equal(np.signbit(dq), np.signbit(v))


def _ue8m0_quant(x):
    with oracle.scale_rule(ue8m0=True):
        return oracle.quant_1x128(x, sc_layout="row_major")


def test_ue8m0_scales_are_the_smallest_unsaturating_powers_of_two():
    """Power-of-two scales (prime-rl PR #4073 conventions table, rows
    "Two-stage weights" and "Compact formats"): every scale is 2^e; the
    tile's absmax stays within the E4M3 range after division (up to the fp32
    rounding of amax / 448 that the rule starts from); half the scale would
    push it past 448; the absmax element encodes to a code in [224, 448];
    and since the quotient v / 2^e is exact, every code is the E4M3 rounding
    of the exact v / s."""
    R, C = 64, 128 * 4
    x = _tile_inputs(R, C, seed=8)
    q, sc = _ue8m0_quant(x)
    t = oracle.e4m3_table().astype(np.float64)
    v = oracle.bf16_to_f32(x).reshape(R, -1, 128).astype(np.float64)
    mant, _ = np.frexp(sc)
    assert np.all(mant == 0.5)
    amax = np.abs(v).max(-1)
    nz = amax > 0
    s = sc.astype(np.float64)
    assert np.all(amax[nz] / s[nz] <= 448.0 * (1 + 2.0 ** -23))
    assert np.all(amax[nz] / (s[nz] / 2) > 448.0 * (1 - 2.0 ** -23))
    assert np.all(sc[~nz] == 1.0)
    dq = t[q].reshape(R, -1, 128)
    top = np.take_along_axis(dq, np.abs(v).argmax(-1)[..., None], -1)[..., 0]
    assert np.all((np.abs(top[nz]) >= 224.0) & (np.abs(top[nz]) <= 448.0))
    exact = (v / s[..., None]).astype(np.float32)          # exact: s is a power of two
    enc = oracle.e4m3_encode_array(exact.ravel()).reshape(exact.shape)
    assert np.array_equal(enc, q.reshape(R, -1, 128))


def test_scale_floors_closed_forms():
    """Floors (prime-rl PR #4073 conventions table, rows "Weight floors" and
    "Activation floors"): an amax floor f gives a zero tile the scale
    fp32(f / 448); a scale floor g gives it g; tiles whose own scale is
    above a floor are unchanged; the UE8M0 rule applies after the floors."""
    x = _tile_inputs(8, 256, seed=9)
    v = oracle.bf16_to_f32(x).reshape(8, -1, 128)
    nz = np.abs(v).max(-1) > 0
    tiny = np.zeros((8, 256), np.uint16)                    # all-zero rows
    _, base = oracle.quant_1x128(x, sc_layout="row_major")
    with oracle.scale_rule(amax_floor=1e-4):
        _, s_a = oracle.quant_1x128(tiny, sc_layout="row_major")
        _, s_ax = oracle.quant_1x128(x, sc_layout="row_major")
    with oracle.scale_rule(scale_floor=2.0 ** -33):
        _, s_s = oracle.quant_1x128(tiny, sc_layout="row_major")
        _, s_sx = oracle.quant_1x128(x, sc_layout="row_major")
    with oracle.scale_rule(ue8m0=True, amax_floor=1e-4):
        _, s_u = oracle.quant_1x128(tiny, sc_layout="row_major")
    assert np.all(s_a == np.float32(np.float32(1e-4) / np.float32(448.0)))
    assert np.all(s_s == np.float32(2.0 ** -33))
    big = nz & (base >= np.float32(1e-4) / np.float32(448.0))
    assert np.array_equal(s_ax[big], base[big]) and np.array_equal(s_sx[big], base[big])
    # 1e-4 / 448 = 2.23e-7 lies in [2^-23, 2^-22): UE8M0 rounds it up to 2^-22
    assert np.all(s_u == np.float32(2.0 ** -22))


def test_philox_known_answers():
    for row in _golden("philox4x32_10_kat.txt"):
        w = [int(v, 16) for v in row]
        assert list(oracle.philox4x32_10(w[0:4], w[4:6])) == w[6:10]


def _sr_example_row():
    x = np.zeros((1, 128), np.float32)
    x[0, :4] = 1.0625
    x[0, 127] = 448.0
    return oracle.f32_to_bf16(x)


def test_sr_worked_example():
    q, sc = oracle.quant_1x128_sr(_sr_example_row(), seed=0, salt=0)
    assert sc[0, 0] == 1.0
    want = {int(r[0]): int(r[1], 16) for r in _golden("sr_worked_example.txt")}
    assert {i: int(q[0, i]) for i in want} == want
    assert q[0, 127] == 0x7E


def test_sr_rule_properties():
    """Values on the E4M3 grid never move; off the grid the result flips from
    the upper to the lower neighbour exactly where the 20-bit fraction stops
    exceeding the random word's top 20 bits; |x| >= 448 saturates; signs and
    signed zeros are kept; the subnormal range uses the 2^-9 grid."""
    t = oracle.e4m3_table()
    rng = np.random.default_rng(3)
    for c in list(range(0x00, 0x7F)):
        for r in rng.integers(0, 2 ** 32, 4, dtype=np.uint64):
            assert oracle.e4m3_encode_sr(float(t[c]), int(r)) == c
            assert oracle.e4m3_encode_sr(-float(t[c]), int(r)) == (c | 0x80)
    # 1 + 3/8 * 2^-3: between 1.0 (0x38) and 1.125 (0x39), F = 0.375 * 2^20
    x = 1.0 + 0.375 * 0.125
    F = int(0.375 * 2 ** 20)
    assert oracle.e4m3_encode_sr(x, (F - 1) << 12) == 0x39
    assert oracle.e4m3_encode_sr(x, F << 12) == 0x38
    assert oracle.e4m3_encode_sr(-x, 0) == 0xB9
    # subnormal range: 2.5 * 2^-9 lies between codes 2 and 3 with F = 2^19
    y = 2.5 * 2.0 ** -9
    assert oracle.e4m3_encode_sr(y, ((1 << 19) - 1) << 12) == 0x03
    assert oracle.e4m3_encode_sr(y, (1 << 19) << 12) == 0x02
    # below the smallest subnormal, including signed zeros
    assert oracle.e4m3_encode_sr(-1e-30, 0xFFFFFFFF) == 0x80
    assert oracle.e4m3_encode_sr(-0.0, 0) == 0x80
    assert oracle.e4m3_encode_sr(1000.0, 0) == 0x7E and oracle.e4m3_encode_sr(-449.0, 0) == 0xFE


def test_sr_is_unbiased():
    """E[dec(q)] equals the quotient up to the 2^-20 cut of the fraction: the
    mean over 4096 rows (independent counters) of one row pattern stays within
    five standard errors of each value."""
    R = 4096
    vals = np.array([1.0625, 1.03, 0.3, -5.7, 100.2, 0.004, -0.0011, 447.0], np.float32)
    x = np.zeros((R, 128), np.float32)
    x[:, :vals.size] = vals
    x[:, 127] = 448.0                                       # scale exactly 1
    xb = oracle.f32_to_bf16(x)
    v = oracle.bf16_to_f32(xb)[0, :vals.size].astype(np.float64)
    q, _ = oracle.quant_1x128_sr(xb, seed=12345, salt=7)
    t = oracle.e4m3_table().astype(np.float64)
    mean = t[q[:, :vals.size]].mean(0)
    for j, xv in enumerate(v):
        lo = t[:0x7F][t[:0x7F] <= abs(xv)].max()
        hi = t[:0x7F][t[:0x7F] > abs(xv)].min() if abs(xv) < 448 else lo
        f = (abs(xv) - lo) / (hi - lo) if hi > lo else 0.0
        se = np.sqrt(f * (1 - f) / R) * (hi - lo)
        assert abs(mean[j] - xv) <= 5 * se + (hi - lo) * 2.0 ** -20 + 1e-12, (j, xv, mean[j])


def _requant_sr_input(R=200, C=64, seed=8):
    """Columns whose token tiles all contain 448 (scale exactly 1) and
    values off the E4M3 grid."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((R, C)) * 20.0).astype(np.float32)
    x[::128, :] = 448.0
    return oracle.f32_to_bf16(x)


def test_requant_sr_brackets_and_scales():
    """The stochastically rounded transposed cast keeps the round-to-nearest
    scales, and every code is one of the two E4M3 neighbours of v / s (the
    same sign), the nearest-rounded code being one of them."""
    xb = _requant_sr_input()
    q0, s0 = oracle.requant_128x1_T(xb)
    q1, s1 = oracle.requant_128x1_T_sr(xb, seed=99, salt=3)
    assert np.array_equal(s0, s1) and np.all(s0 == 1.0)
    t = oracle.e4m3_table().astype(np.float64)
    v = oracle.bf16_to_f32(xb).astype(np.float64).T          # [C x R], scale 1
    R = v.shape[1]
    a = np.abs(v)
    pos = t[:0x7F]
    lo = np.array([[pos[pos <= e].max() for e in row] for row in a])
    hi = np.array([[pos[pos >= e].min() if e <= 448 else 448.0 for e in row] for row in a])
    got = np.abs(t[q1[:, :R]])
    assert np.all((got == lo) | (got == hi))
    assert np.all(np.signbit(t[q1[:, :R]]) == np.signbit(v))
    near = np.abs(t[q0[:, :R]])
    assert np.all((near == lo) | (near == hi))
    assert np.all(q1[:, R:] == 0)                            # padding tokens


def test_requant_sr_word_per_source_element():
    """Element (r, c) of the source takes the random word of index r * C + c:
    with scale 1 the transposed SR codes equal the pinned SR encoder applied
    with those words, and a shifted index mapping disagrees."""
    xb = _requant_sr_input(R=130, C=32, seed=9)
    q, _ = oracle.requant_128x1_T_sr(xb, seed=5, salt=11)
    v = oracle.bf16_to_f32(xb)
    R, C = v.shape
    want = np.array([[oracle.e4m3_encode_sr(float(v[r, c]), oracle.sr_word(5, 11, r * C + c))
                      for r in range(R)] for c in range(C)], np.uint8)
    assert np.array_equal(q[:, :R], want)
    shifted = np.array([[oracle.e4m3_encode_sr(float(v[r, c]), oracle.sr_word(5, 11, c * R + r))
                         for r in range(R)] for c in range(C)], np.uint8)
    assert not np.array_equal(q[:, :R], shifted)


def test_requant_sr_is_unbiased():
    """Identical columns (independent counters) average to v / s within five
    standard errors."""
    C = 4096
    vals = np.array([1.0625, 1.03, 0.3, -5.7, 100.2, 0.004, -0.0011, 447.0], np.float32)
    x = np.zeros((128, C), np.float32)
    x[:vals.size, :] = vals[:, None]
    x[127, :] = 448.0
    xb = oracle.f32_to_bf16(x)
    v = oracle.bf16_to_f32(xb)[:vals.size, 0].astype(np.float64)
    q, s = oracle.requant_128x1_T_sr(xb, seed=2024, salt=1)
    assert np.all(s == 1.0)
    t = oracle.e4m3_table().astype(np.float64)
    mean = t[q[:, :vals.size]].mean(0)
    for j, xv in enumerate(v):
        lo = t[:0x7F][t[:0x7F] <= abs(xv)].max()
        hi = t[:0x7F][t[:0x7F] > abs(xv)].min() if abs(xv) < 448 else lo
        f = (abs(xv) - lo) / (hi - lo) if hi > lo else 0.0
        se = np.sqrt(f * (1 - f) / C) * (hi - lo)
        assert abs(abs(mean[j]) - abs(xv)) <= 5 * se + (hi - lo) * 2.0 ** -20 + 1e-12, (j, xv, mean[j])


def _philox_word(seed, salt, idx):
    """The random word of element idx, restated from the Philox4x32-10 block
    function that the published known-answer vectors pin: counter (idx / 4
    low, idx / 4 high, salt, 0), key (seed low, seed high), output word
    idx % 4."""
    c = idx // 4
    out = oracle.philox4x32_10([c & 0xFFFFFFFF, c >> 32, salt & 0xFFFFFFFF, 0],
                               [seed & 0xFFFFFFFF, seed >> 32])
    return int(out[idx % 4])


def _sr128_input():
    """Rows of widely different magnitude (so the three column blocks and the
    two row blocks get different scales); 128 + 16 rows leave a ragged row
    block."""
    rng = np.random.default_rng(31)
    R, C = 128 + 16, 384
    x = (rng.standard_normal((R, C)) * np.exp(rng.uniform(-3.0, 3.0, (R, 1)))).astype(np.float32)
    return oracle.f32_to_bf16(x)


def test_quant_128x128_sr_word_per_tensor_element():
    """128x128 cast with stochastic rounding (prime-rl PR #4073, "SR agreement"
    row; reading: element (r, c) of matrix b of a batch of R x C matrices takes
    the word of index b R C + r C + c). Every code is the pinned SR encoder
    applied to the fp32 quotient v / s, s being the round-to-nearest cast's
    block scale, with the word restated from the pinned Philox function; a
    block-local or a transposed element numbering disagrees."""
    xb = _sr128_input()
    v = oracle.bf16_to_f32(xb)
    R, C = v.shape
    seed, salt = 0x123456789ABC, 7
    _, s_rn = oracle.quant_128x128(xb)
    s_el = np.repeat(np.repeat(s_rn, 128, 0), 128, 1)[:R, :C]
    quot = (v / s_el).astype(np.float32)              # IEEE fp32 division, round to nearest
    for b in range(2):
        base = b * R * C
        q, s = oracle.quant_128x128_sr(xb, seed=seed, salt=salt, idx_base=base)
        assert np.array_equal(s.view(np.uint32), s_rn.view(np.uint32))
        want = np.array([[oracle.e4m3_encode_sr(float(quot[r, c]), _philox_word(seed, salt, base + r * C + c))
                          for c in range(C)] for r in range(R)], np.uint8)
        assert np.array_equal(q, want)
    # the numbering matters: block-local and transposed indices give other codes
    rows = range(4)
    block_local = np.array([[oracle.e4m3_encode_sr(
        float(quot[r, c]), _philox_word(seed, salt, (c // 128) * 128 * 128 + r * 128 + c % 128))
        for c in range(C)] for r in rows], np.uint8)
    transposed = np.array([[oracle.e4m3_encode_sr(float(quot[r, c]), _philox_word(seed, salt, c * R + r))
                            for c in range(C)] for r in rows], np.uint8)
    q0, _ = oracle.quant_128x128_sr(xb, seed=seed, salt=salt)
    assert not np.array_equal(q0[:4], block_local)
    assert not np.array_equal(q0[:4], transposed)


def _mode_q_input():
    """An E4M3 stash [300 x 256] with random finite codes (a row of -0 codes
    and a zero tile included) and 1x128 scales that differ for every row and
    column tile."""
    rng = np.random.default_rng(32)
    M, C = 300, 256
    t = oracle.e4m3_table()
    fin = np.nonzero(~np.isnan(t))[0]
    q = rng.choice(fin, size=(M, C)).astype(np.uint8)
    q[5, :] = 0x80
    q[256:, 128:] = 0x00
    sc = (np.exp2(rng.integers(-12, 4, (C // 128, M))) * rng.uniform(1.0, 2.0, (C // 128, M))).astype(np.float32)
    ld = oracle.scale_rows_padded(M)
    sc_tm = np.zeros((C // 128, ld), np.float32)
    sc_tm[:, :M] = sc
    return q, sc_tm


def test_requant_mode_q_varying_scales_matches_torch_steps():
    """E4M3-source 128x1 requant ("scratch: the backward pass, unrolled",
    "What is asserted, and from where", bullet 2: the Wgrad operands are
    re-tiled 128x1 from the saved tensors). Reading: each saved code is
    decoded as fp32(dec(q) * s) with the 1x128 scale of its own row and
    column tile, then quantized along tokens. Restated here with torch's own
    E4M3 decoding, a numpy fp32 multiply and the torch-steps quantizer on the
    transposed operand, with scales that differ for every row and tile;
    dense and grouped (an empty group and a group of one tile + 1 token)."""
    q, sc = _mode_q_input()
    M, C = q.shape
    dec = torch.from_numpy(q).view(torch.float8_e4m3fn).float().numpy()
    s_el = np.repeat(sc[:, :M].T, 128, axis=1)
    deq = (dec * s_el).astype(np.float32)             # one fp32 multiply per element
    for offsets in (None, [0, 129, 129, 300]):
        qT, scT = oracle.requant_128x1_T(q, sc, offsets=offsets)
        segs = [(0, M)] if offsets is None else list(zip(offsets[:-1], offsets[1:]))
        p = 0
        for a, b in segs:
            for t0 in range(a, b, 128):
                n = min(t0 + 128, b) - t0
                qr, sr = _torch_quant_rows(np.ascontiguousarray(deq[t0:t0 + n, :].T))
                assert np.array_equal(qT[:, p:p + n], qr)
                assert np.all(qT[:, p + n:p + 128] == 0)
                assert np.array_equal(scT[p // 128].view(np.uint32), sr.view(np.uint32))
                p += 128
        assert p == qT.shape[1]


def test_mx_quant_scales_and_codes():
    """MXFP8 (OCP MX v1.0 blocks of 32 with 8-bit exponent scales): each
    scale 2^(E-127) is the smallest power of two that keeps the block's
    absmax within 448 (up to the fp32 rounding of amax / 448); a zero block
    has E = 127; every code is the E4M3 rounding of the exact v / 2^(E-127)."""
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((16, 256)) * np.exp(rng.uniform(-8, 8, (16, 1)))).astype(np.float32)
    x[3, 32:64] = 0.0
    xb = oracle.f32_to_bf16(x)
    q, E = oracle.mx_quant_1x32(xb)
    v = oracle.bf16_to_f32(xb).astype(np.float64).reshape(16, 8, 32)
    amax = np.abs(v).max(-1)
    X = np.ldexp(1.0, E.astype(np.int64) - 127)
    nz = amax > 0
    assert np.all(E[~nz] == 127)
    assert np.all(amax[nz] / X[nz] <= 448.0 * (1 + 2.0 ** -23))
    assert np.all(amax[nz] / (X[nz] / 2) > 448.0 * (1 - 2.0 ** -23))
    exact = (v / X[..., None]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode_array(exact.ravel()).reshape(16, 256), q)


def test_mx_gemm_vs_fp64_dequantized():
    """The MXFP8 GEMM equals the fp64 product of the dequantized operands up
    to one fp32 rounding."""
    rng = np.random.default_rng(5)
    M, N, K = 48, 40, 512
    a = oracle.f32_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    b = oracle.f32_to_bf16((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    qa, ea = oracle.mx_quant_1x32(a)
    qb, eb = oracle.mx_quant_1x32(b)
    t = oracle.e4m3_table().astype(np.float64)
    da = t[qa] * np.repeat(np.ldexp(1.0, ea.astype(np.int64) - 127), 32, 1)
    db = t[qb] * np.repeat(np.ldexp(1.0, eb.astype(np.int64) - 127), 32, 1)
    truth = da @ db.T
    out = oracle.mx_gemm(qa, ea, qb, eb)
    bound = 2.0 ** -23 * np.abs(truth) + 1e-12 * (np.abs(da) @ np.abs(db).T)
    assert np.all(np.abs(out - truth) <= bound)
    ii, jj = np.array([0, 7, 47]), np.array([39, 3, 0])
    assert np.array_equal(oracle.mx_gemm(qa, ea, qb, eb, ii, jj), out[ii, jj])


def test_quant_reciprocal_case_is_distinguished():
    """A tile where v * (1/s) and v / s round to different E4M3 codes: the
    torch-steps pin must see the true division."""
    v = _find_reciprocal_mismatch()
    x = oracle.f32_to_bf16(v.reshape(1, 128))
    q, sc = oracle.quant_1x128(x, sc_layout="row_major")
    qr, sr = _torch_quant_rows(oracle.bf16_to_f32(x))
    assert np.array_equal(q, qr) and sc[0, 0] == sr[0]


def _find_reciprocal_mismatch():
    """Search bf16 tiles (amax and one probe value) until fp32 division and
    multiplication by the fp32 reciprocal give different E4M3 codes."""
    g = np.random.default_rng(7)
    amaxes = oracle.bf16_to_f32(oracle.f32_to_bf16(g.uniform(1.0, 1000.0, 4000).astype(np.float32)))
    probes = oracle.bf16_to_f32(np.arange(0x3C00, 0x4400, dtype=np.uint16))
    for a in amaxes:
        s = np.float32(a) / np.float32(448.0)
        d = _torch_cast_codes(probes / s)
        m = _torch_cast_codes(probes * (np.float32(1.0) / s))
        bad = np.nonzero(d != m)[0]
        if bad.size:
            v = np.zeros(128, np.float32)
            v[0] = a
            v[1] = probes[bad[0]]
            return v
    raise AssertionError("no mismatching case found")


def test_requant_mode_b_is_1x128_of_transpose():
    """128x1 tiles of X along tokens = 1x128 tiles of X^T along its rows."""
    M, C = 300, 200
    x = _tile_inputs(M, C, seed=8)
    qT, scT = oracle.requant_128x1_T(x)
    q1, s1 = oracle.quant_1x128(np.ascontiguousarray(x.T), sc_layout="row_major")
    mp = oracle.padded_tokens(M)
    assert qT.shape == (C, mp) and scT.shape == (mp // 128, C)
    assert np.array_equal(qT[:, :M], q1)
    assert np.all(qT[:, M:] == 0)
    assert np.array_equal(scT.T, s1)


def test_requant_mode_q_power_of_two_is_transpose():
    """If a 128x128 block's 1x128 scales are one power of two and every token
    column holds a +-448 code, the 128x1 requant keeps the scale and the
    payload is the byte transpose."""
    g = np.random.default_rng(9)
    M, C = 256, 256
    t = oracle.e4m3_table()
    fin = np.nonzero(~np.isnan(t))[0]
    q = g.choice(fin, size=(M, C)).astype(np.uint8)
    for tile in range(M // 128):
        rows = tile * 128 + g.integers(0, 128, size=C)
        q[rows, np.arange(C)] = np.where(g.random(C) < 0.5, 0x7E, 0xFE)
    s = np.float32(2.0 ** -7)
    sc = np.full((C // 128, M), s, np.float32)
    qT, scT = oracle.requant_128x1_T(q, sc)
    assert np.all(scT == s)
    assert np.array_equal(qT, q.T)


def test_requant_groups_geometry_and_padding():
    M, C = 400, 128
    counts = [0, 129, 1, 0, 270]
    off = wl.offsets_from_counts(counts)
    x = _tile_inputs(M, C, seed=10)
    qT, scT = oracle.requant_128x1_T(x, offsets=off)
    mp = sum(-(-n // 128) * 128 for n in counts)
    assert qT.shape == (C, mp) and scT.shape == (mp // 128, C)
    p = 0
    for e, n in enumerate(counts):
        if n == 0:
            continue
        seg = np.ascontiguousarray(x[off[e]:off[e + 1]])
        qe, se = oracle.requant_128x1_T(seg)
        w = qe.shape[1]
        assert np.array_equal(qT[:, p:p + w], qe)
        assert np.array_equal(scT[p // 128:(p + w) // 128], se)
        p += w


# ---------------------------------------------------------------------------
# Promoted GEMMs against fp64 of the dequantized operands
# ---------------------------------------------------------------------------

def _deq_rows(q, sc_row_major, tile_axis_len=128):
    t = oracle.e4m3_table().astype(np.float64)
    v = t[q]
    s = np.repeat(sc_row_major.astype(np.float64), tile_axis_len, axis=1)[:, :q.shape[1]]
    return v * s


def _deq_blocks(q, sc):
    t = oracle.e4m3_table().astype(np.float64)
    s = np.repeat(np.repeat(sc.astype(np.float64), 128, 0), 128, 1)[:q.shape[0], :q.shape[1]]
    return t[q] * s


def _bound(absprod, nblocks):
    return (nblocks + 3) * 2.0 ** -23 * absprod + 1e-30


def _fprop_case(M, K, N, seed):
    x = _tile_inputs(M, K, seed)
    w = wl.bits(wl.normal((K, N), std=0.02, seed=seed + 50))
    xq, sx = oracle.quant_1x128(x)
    wq, sw = oracle.quant_128x128(w)
    return xq, sx, wq, sw


def _check_fprop(M, K, N, seed):
    xq, sx, wq, sw = _fprop_case(M, K, N, seed)
    y = oracle.fprop(xq, sx, wq, sw)
    a = _deq_rows(xq, np.ascontiguousarray(sx[:, :M].T))
    b = _deq_blocks(wq, sw)
    ref = a @ b
    absprod = np.abs(a) @ np.abs(b)
    return np.all(np.abs(y - ref) <= _bound(absprod, -(-K // 128)))


@pytest.mark.parametrize("M,K,N", [(3, 128, 128), (130, 384, 256), (64, 200, 136)])
def test_fprop_vs_fp64_dequantized(M, K, N):
    assert _check_fprop(M, K, N, seed=11)


def _check_dgrad(M, N, K, seed):
    dy = _tile_inputs(M, N, seed)
    w = wl.bits(wl.normal((K, N), std=0.02, seed=seed + 60))
    dyq, sdy = oracle.quant_1x128(dy)
    wq, sw = oracle.quant_128x128(w)
    dx = oracle.dgrad(dyq, sdy, wq, sw)
    a = _deq_rows(dyq, np.ascontiguousarray(sdy[:, :M].T))
    b = _deq_blocks(wq, sw)
    ref = a @ b.T
    absprod = np.abs(a) @ np.abs(b).T
    return np.all(np.abs(dx - ref) <= _bound(absprod, -(-N // 128)))


@pytest.mark.parametrize("M,N,K", [(5, 256, 128), (129, 384, 256)])
def test_dgrad_vs_fp64_dequantized(M, N, K):
    assert _check_dgrad(M, N, K, seed=12)


def _check_wgrad(T, N, K, seed):
    dy = _tile_inputs(T, N, seed)
    x = _tile_inputs(T, K, seed + 1)
    dyqT, sdyT = oracle.requant_128x1_T(dy)
    xqT, sxT = oracle.requant_128x1_T(x)
    dw = oracle.wgrad(dyqT, sdyT, xqT, sxT)
    t = oracle.e4m3_table().astype(np.float64)
    a = t[dyqT] * np.repeat(sdyT.T.astype(np.float64), 128, axis=1)   # [N x Tpad]
    b = t[xqT] * np.repeat(sxT.T.astype(np.float64), 128, axis=1)     # [K x Tpad]
    ref = a @ b.T
    absprod = np.abs(a) @ np.abs(b).T
    return np.all(np.abs(dw - ref) <= _bound(absprod, dyqT.shape[1] // 128))


@pytest.mark.parametrize("T,N,K", [(128, 128, 256), (300, 256, 128)])
def test_wgrad_vs_fp64_dequantized(T, N, K):
    assert _check_wgrad(T, N, K, seed=13)


def test_single_block_reduces_to_plain_dot():
    """One K-block with unit scales: the promoted GEMM is the plain dot
    product of the decoded codes, which is exact in fp32 here."""
    g = np.random.default_rng(14)
    t = oracle.e4m3_table()
    small = np.nonzero((~np.isnan(t)) & (np.abs(t) <= 4) & (np.abs(t) >= 2 ** -3))[0]
    xq = g.choice(small, size=(8, 128)).astype(np.uint8)
    wq = g.choice(small, size=(128, 16)).astype(np.uint8)
    sx = np.ones((1, 8), np.float32)
    sw = np.ones((1, 1), np.float32)
    y = oracle.fprop(xq, sx, wq, sw)
    ref = t[xq].astype(np.float64) @ t[wq].astype(np.float64)
    assert np.array_equal(y, ref.astype(np.float32))


def test_fprop_sampled_elements_match_full():
    xq, sx, wq, sw = _fprop_case(70, 256, 256, seed=15)
    full = oracle.fprop(xq, sx, wq, sw)
    ii = np.array([0, 69, 33, 5]); jj = np.array([255, 0, 128, 17])
    assert np.array_equal(oracle.fprop(xq, sx, wq, sw, ii, jj), full[ii, jj])


def test_grouped_fprop_is_per_expert_dense():
    counts = [3, 0, 130]
    off = wl.offsets_from_counts(counts)
    M, K, N = sum(counts), 256, 128
    x = _tile_inputs(M, K, 16)
    xq, sx = oracle.quant_1x128(x)
    ws = [oracle.quant_128x128(wl.bits(wl.normal((K, N), 0.02, seed=17 + e))) for e in range(3)]
    wq = np.stack([w[0] for w in ws]); sw = np.stack([w[1] for w in ws])
    y = oracle.grouped_fprop(xq, sx, wq, sw, off)
    for e in range(3):
        r0, r1 = off[e], off[e + 1]
        if r1 > r0:
            a = _deq_rows(xq[r0:r1], np.ascontiguousarray(sx[:, r0:r1].T))
            ref = a @ _deq_blocks(wq[e], sw[e])
            assert np.allclose(y[r0:r1], ref, rtol=1e-5, atol=1e-6)


# ---------------------------------------------------------------------------
# Drift (partial-sum page, sections 2, 4 and 5)
# ---------------------------------------------------------------------------

def test_round_sig_closed_forms():
    assert oracle.round_sig(1.0 + 2 ** -20, 14) == 1.0
    assert oracle.round_sig(1.0 + 3 * 2 ** -14, 14) == 1.0 + 4 * 2 ** -14   # tie to even
    assert oracle.round_sig(1.0 + 2 ** -14, 14) == 1.0                      # tie to even
    assert oracle.round_sig(1.999, 8, mode=1) == 1.9921875                  # toward zero
    assert oracle.round_sig(-3.0, 1) == -4.0


@pytest.mark.slow
def test_drift_grows_with_k_only_without_promotion():
    promoted, unpromoted = [], []
    ii = np.arange(8) * 31 % 256
    jj = np.arange(8) * 17 % 256
    for K in wl.LONGK_VALUES:
        d = wl.longk(K)
        xq, sx = oracle.quant_1x128(wl.bits(d["X"]))
        wq, sw = oracle.quant_128x128(wl.bits(d["W"]))
        y = oracle.fprop(xq, sx, wq, sw, ii, jj).astype(np.float64)
        truth, unpr = oracle.fprop_reference_sums(xq, sx, wq, sw, ii, jj, m_bits=14)
        promoted.append(np.max(np.abs(y - truth) / np.abs(truth)))
        unpromoted.append(np.max(np.abs(unpr - truth) / np.abs(truth)))
    promoted, unpromoted = np.array(promoted), np.array(unpromoted)
    assert np.all(promoted < 1e-6)                   # bounded by fp32 rounding
    assert np.all(np.diff(unpromoted) > 0)           # grows with K
    assert unpromoted[-1] > 1e-2                     # stagnation at K = 65536
    ratio = unpromoted / np.maximum(promoted, 1e-12)
    assert np.all(np.diff(ratio) > 0)


# ---------------------------------------------------------------------------
# Negative controls: each planted mistake must make a pin fail
# ---------------------------------------------------------------------------

def _pin_encoder():
    try:
        test_encoder_golden_cases()
        return True
    except AssertionError:
        return False


def _pin_quant():
    try:
        test_quant_1x128_matches_torch_steps()
        test_quant_reciprocal_case_is_distinguished()
        return True
    except AssertionError:
        return False


def _pin_scale_rules():
    try:
        test_ue8m0_scales_are_the_smallest_unsaturating_powers_of_two()
        test_scale_floors_closed_forms()
        return True
    except AssertionError:
        return False


def _pin_sr():
    try:
        test_sr_worked_example()
        test_sr_is_unbiased()
        return True
    except AssertionError:
        return False


def _pin_sr128():
    try:
        test_quant_128x128_sr_word_per_tensor_element()
        return True
    except AssertionError:
        return False


def _pin_requant_q():
    try:
        test_requant_mode_q_varying_scales_matches_torch_steps()
        return True
    except AssertionError:
        return False


def _pin_gemm():
    return (_check_fprop(130, 384, 256, 21) and _check_dgrad(129, 384, 256, 22)
            and _check_wgrad(300, 256, 128, 23) and _check_fprop(64, 256, 256, 24))


@pytest.mark.parametrize("fault,pin", [
    (oracle.FAULT_DROP_LAST_BLOCK, "gemm"),
    (oracle.FAULT_SCALE_NEXT_BLOCK, "gemm"),
    (oracle.FAULT_TIES_AWAY, "encoder"),
    (oracle.FAULT_SIGNED_AMAX, "quant"),
    (oracle.FAULT_TRANSPOSED_W, "gemm"),
    (oracle.FAULT_DROP_NEG_ZERO, "encoder"),
    (oracle.FAULT_RECIPROCAL, "quant"),
    (oracle.FAULT_SIGN_FLIP_TERM, "gemm"),
    (oracle.FAULT_UE8M0_DOWN, "scale_rules"),
    (oracle.FAULT_FLOOR_AFTER, "scale_rules"),
    (oracle.FAULT_SR_WORD, "sr"),
    (oracle.FAULT_SR_NEAREST, "sr"),
    (oracle.FAULT_SR_BLOCK_INDEX, "sr128"),
    (oracle.FAULT_REQUANT_TILE_SCALE, "requant_q"),
])
def test_planted_mistake_is_caught(fault, pin):
    check = {"encoder": _pin_encoder, "quant": _pin_quant, "gemm": _pin_gemm,
             "scale_rules": _pin_scale_rules, "sr": _pin_sr, "sr128": _pin_sr128,
             "requant_q": _pin_requant_q}[pin]
    assert check()
    oracle.set_fault(fault)
    try:
        assert not check()
    finally:
        oracle.set_fault(oracle.FAULT_NONE)
    assert check()


# ---------------------------------------------------------------------------
# Packed exponent bytes of power-of-two scales (prime-rl PR #4073 conventions
# table, row "Compact formats"; OCP MX v1.0 exponent-byte format)
# ---------------------------------------------------------------------------

def test_pack_ue8m0_exponent_bytes_closed_form():
    """Every exponent byte E in 0..254 is the byte of the scale 2^(E - 127)
    (2^-127 is an fp32 subnormal and still has one); every K-block's byte
    covers its four 32-element blocks; anything that is not a positive power
    of two in [2^-127, 2^127] has no byte (255) and is counted."""
    E = np.arange(255)
    s = np.ldexp(1.0, E - 127).astype(np.float32)
    assert np.array_equal(s.astype(np.float64), np.ldexp(1.0, E - 127))   # all exact in fp32
    b, bad = oracle.pack_ue8m0(s, 255, 256, 1, 1, 0)
    assert bad == 0 and b.shape == (255, 8)
    assert np.array_equal(b[:, 0], E) and (b == b[:, :1]).all()
    odd = np.array([0.75, 3.0, 0.0, -1.0, -0.5, np.inf, np.nan, 2.0 ** -128, 2.0 ** -149,
                    np.float32(1.0) + np.float32(2.0 ** -23)], np.float32)
    b, bad = oracle.pack_ue8m0(odd, odd.size, 128, 1, 1, 0)
    assert bad == odd.size and (b == 255).all()


def _ue8m0_operands(M=200, K=384, N=256, seed=5):
    rng = np.random.default_rng(seed)
    x = oracle.f32_to_bf16((rng.standard_normal((M, K)) * np.exp(2 * rng.standard_normal((M, 1)))).astype(np.float32))
    w = oracle.f32_to_bf16((rng.standard_normal((K, N)) * 0.02).astype(np.float32))
    with oracle.scale_rule(ue8m0=True):
        xq, sx = oracle.quant_1x128(x)
        wq, sw = oracle.quant_128x128(w)
        xT, sxT = oracle.requant_128x1_T(xq, sx)
    return xq, sx, wq, sw, xT, sxT


def _mx_dequant(q, e):
    """Values of an MX operand: E4M3 codes times 2^(E - 127) per 32-element block."""
    return oracle.e4m3_decode(q).astype(np.float64) * np.ldexp(1.0, np.repeat(e.astype(np.int64) - 127, 32, axis=1))


def test_pack_ue8m0_reproduces_the_block_dequantization():
    """With UE8M0-rule scales, dequantizing through the packed bytes (per
    32-element block) gives exactly the 1x128 / 128x128 dequantization (per
    128-element block) for the four operand layouts: activation rows, the
    transposed 128x1 operand, W^T (Fprop's B) and W (Dgrad's B); a ragged
    row count and a wrong stride are both caught."""
    M, K, N = 200, 384, 256
    xq, sx, wq, sw, xT, sxT = _ue8m0_operands(M, K, N)
    dec = lambda q: oracle.e4m3_decode(q).astype(np.float64)
    # activation rows: scale (r, b) = sx[b, r]
    b, bad = oracle.pack_ue8m0(sx, M, K, 1, 1, sx.shape[1])
    assert bad == 0
    assert np.array_equal(_mx_dequant(xq, b), dec(xq) * np.repeat(sx[:, :M].T, 128, axis=1))
    # transposed operand [K x Mpad]: scale (k, token block t) = sxT[t, k]
    Mp = xT.shape[1]
    b, bad = oracle.pack_ue8m0(sxT, K, Mp, 1, 1, K)
    assert bad == 0
    assert np.array_equal(_mx_dequant(xT, b), dec(xT) * np.repeat(sxT.T, 128, axis=1))
    # W^T [N x K]: scale (n, b) = sw[b, n // 128]
    wT = np.ascontiguousarray(wq.T)
    b, bad = oracle.pack_ue8m0(sw, N, K, 128, 1, N // 128)
    assert bad == 0
    assert np.array_equal(_mx_dequant(wT, b), dec(wT) * np.repeat(np.repeat(sw.T, 128, axis=0), 128, axis=1))
    # W [K x N] with the contraction along N: scale (k, nb) = sw[k // 128, nb]
    b, bad = oracle.pack_ue8m0(sw, K, N, 128, N // 128, 1)
    assert bad == 0
    assert np.array_equal(_mx_dequant(wq, b), dec(wq) * np.repeat(np.repeat(sw, 128, axis=0), 128, axis=1))
    # a wrong stride (the row pitch of the 1x128 array off by one) is not the same operand
    b, _ = oracle.pack_ue8m0(sx, M, K, 1, 1, sx.shape[1] - 1)
    assert not np.array_equal(_mx_dequant(xq, b), dec(xq) * np.repeat(sx[:, :M].T, 128, axis=1))


def test_pack_ue8m0_mx_gemm_is_the_promoted_gemm():
    """The oracle's MX GEMM over packed UE8M0 operands agrees with the
    oracle's per-128 promoted Fprop to fp32 summation-order accuracy: with
    power-of-two scales the block scaling of the tensor core computes the
    recipe's GEMM, only the order of the fp32 additions differs."""
    M, K, N = 200, 384, 256
    xq, sx, wq, sw, _, _ = _ue8m0_operands(M, K, N)
    bx, _ = oracle.pack_ue8m0(sx, M, K, 1, 1, sx.shape[1])
    bw, _ = oracle.pack_ue8m0(sw, N, K, 128, 1, N // 128)
    y_mx = oracle.mx_gemm(xq, bx, np.ascontiguousarray(wq.T), bw).astype(np.float64)
    y_pr = oracle.fprop(xq, sx, wq, sw).astype(np.float64)
    a = np.abs(_mx_dequant(xq, bx))
    bt = np.abs(_mx_dequant(np.ascontiguousarray(wq.T), bw))
    absprod = a @ bt.T
    assert np.all(np.abs(y_mx - y_pr) <= 2.0 ** -20 * absprod + 1e-30)
    assert np.count_nonzero(y_pr) > 0.99 * y_pr.size


def test_pack_ue8m0_mx_gemm_is_the_promoted_dgrad_and_wgrad():
    """The same agreement for Dgrad (A = dY rows, B = W with the contraction
    along N) and Wgrad (A = dY^T, B = X^T from the transposed casts): the
    oracle's MX GEMM over the packed operands matches its promoted GEMM to
    fp32 summation-order accuracy, so the stride and row-block choices of
    the packing are the ones each operand needs."""
    rng = np.random.default_rng(11)
    M, K, N = 256, 384, 256
    x = oracle.f32_to_bf16((rng.standard_normal((M, K)) * np.exp(rng.standard_normal((M, 1)))).astype(np.float32))
    w = oracle.f32_to_bf16((rng.standard_normal((K, N)) * 0.02).astype(np.float32))
    dy = oracle.f32_to_bf16((rng.standard_normal((M, N)) * 1e-3).astype(np.float32))
    with oracle.scale_rule(ue8m0=True):
        xq, sx = oracle.quant_1x128(x)
        wq, sw = oracle.quant_128x128(w)
        dyq, sdy = oracle.quant_1x128(dy)
        xT, sxT = oracle.requant_128x1_T(xq, sx)
        dyT, sdyT = oracle.requant_128x1_T(dy)
    Mp = xT.shape[1]
    # Dgrad: dX [M x K] = dY W^T
    ba, _ = oracle.pack_ue8m0(sdy, M, N, 1, 1, sdy.shape[1])
    bb, _ = oracle.pack_ue8m0(sw, K, N, 128, N // 128, 1)
    got = oracle.mx_gemm(dyq, ba, wq, bb).astype(np.float64)
    ref = oracle.dgrad(dyq, sdy, wq, sw).astype(np.float64)
    absprod = np.abs(_mx_dequant(dyq, ba)) @ np.abs(_mx_dequant(wq, bb)).T
    assert np.all(np.abs(got - ref) <= 2.0 ** -20 * absprod + 1e-30)
    # Wgrad: dW [N x K] = dY^T X over the padded tokens
    ba, _ = oracle.pack_ue8m0(sdyT, N, Mp, 1, 1, N)
    bb, _ = oracle.pack_ue8m0(sxT, K, Mp, 1, 1, K)
    got = oracle.mx_gemm(dyT, ba, xT, bb).astype(np.float64)
    ref = oracle.wgrad(dyT, sdyT, xT, sxT).astype(np.float64)
    absprod = np.abs(_mx_dequant(dyT, ba)) @ np.abs(_mx_dequant(xT, bb)).T
    assert np.all(np.abs(got - ref) <= 2.0 ** -20 * absprod + 1e-30)
    # the transposed operand's per-row scales packed as if they were 128-row
    # block scales (a plausible mix-up of the layouts) is not the same GEMM
    bad, _ = oracle.pack_ue8m0(sxT, K, Mp, 128, 1, K)
    assert not np.allclose(oracle.mx_gemm(dyT, ba, xT, bad), ref, rtol=1e-3, atol=0)
