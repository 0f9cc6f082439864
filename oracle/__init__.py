"""CPU oracle for the fine-grained FP8 linear layer (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers. The product path (the CUDA
library and its Python binding) never imports this package.

The arithmetic lives in ``fp8bs_oracle.c`` (plain C99, compiled here with gcc,
no code shared with the CUDA library). This module only compiles it, loads it
with ctypes and marshals numpy arrays. Grouped (MoE) variants loop over the
experts and call the dense routines on each expert's rows, which is the
definition of a grouped GEMM.

Array conventions: bf16 tensors are numpy ``uint16`` arrays holding the bf16
bit patterns; E4M3 payloads are ``uint8``; scales are ``float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8bs_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# planted-mistake switch values (see fp8bs_oracle.c); tests only
FAULT_NONE = 0
FAULT_DROP_LAST_BLOCK = 1
FAULT_SCALE_NEXT_BLOCK = 2
FAULT_TIES_AWAY = 3
FAULT_SIGNED_AMAX = 4
FAULT_TRANSPOSED_W = 5
FAULT_DROP_NEG_ZERO = 6
FAULT_RECIPROCAL = 7
FAULT_SIGN_FLIP_TERM = 8
FAULT_UE8M0_DOWN = 9
FAULT_FLOOR_AFTER = 10
FAULT_SR_WORD = 11
FAULT_SR_NEAREST = 12
FAULT_SR_BLOCK_INDEX = 13
FAULT_REQUANT_TILE_SCALE = 14


def build(force: bool = False) -> str:
    """Compile the oracle library (gcc, -O2, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:-3] + ["-fopenmp"] + base[-3:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # no OpenMP runtime: single-threaded build gives identical results
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.oracle_e4m3_table.argtypes = [P]
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode_array.argtypes = [P, I64, P]
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_float
        lib.oracle_f32_to_bf16_array.argtypes = [P, I64, P]
        lib.oracle_quant_1x128.argtypes = [P, I64, I64, I64, P, I64, P, I64, I64]
        lib.oracle_quant_128x128.argtypes = [P, I64, I64, I64, P, I64, P, I64]
        lib.oracle_padded_tokens.argtypes = [P, I, I64]
        lib.oracle_padded_tokens.restype = I64
        lib.oracle_requant_128x1_T.argtypes = [I, P, I64, P, I64, I64, I64, I64,
                                               P, I, P, I64, P, I64]
        lib.oracle_fprop.argtypes = [P, I64, P, I64, I64, P, I64, P, I64,
                                     I64, I64, I64, P, P, I64, P]
        lib.oracle_dgrad.argtypes = [P, I64, P, I64, I64, P, I64, P, I64,
                                     I64, I64, I64, P, P, I64, P]
        lib.oracle_wgrad.argtypes = [P, I64, P, I64, P, I64, P, I64,
                                     I64, I64, I64, P, P, I64, P]
        lib.oracle_round_sig.argtypes = [ctypes.c_double, I, I]
        lib.oracle_round_sig.restype = ctypes.c_double
        lib.oracle_fprop_reference_sums.argtypes = [P, I64, P, I64, I64, P, I64, P, I64,
                                                    I64, P, P, I64, I, I, P, P]
        lib.oracle_num_threads.restype = I
        lib.oracle_set_num_threads.argtypes = [I]
        lib.oracle_set_fault.argtypes = [I]
        lib.oracle_set_scale_rule.argtypes = [I, ctypes.c_float, ctypes.c_float]
        U32, U64 = ctypes.c_uint32, ctypes.c_uint64
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_sr_word.argtypes = [U64, U32, U64]
        lib.oracle_sr_word.restype = U32
        lib.oracle_e4m3_encode_sr.argtypes = [ctypes.c_float, U32]
        lib.oracle_e4m3_encode_sr.restype = ctypes.c_uint8
        lib.oracle_quant_1x128_sr.argtypes = [P, I64, I64, I64, P, I64, P, I64, I64, U64, U32]
        lib.oracle_requant_128x1_T_sr.argtypes = [I, P, I64, P, I64, I64, I64, I64,
                                                  P, I, P, I64, P, I64, U64, U32]
        lib.oracle_quant_128x128_sr.argtypes = [P, I64, I64, I64, P, I64, P, I64, U64, U32, I64]
        lib.oracle_mx_quant_1x32.argtypes = [P, I64, I64, P, P]
        lib.oracle_mx_gemm.argtypes = [P, P, P, P, I64, I64, I64, P, P, P, I64]
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def set_fault(f: int) -> None:
    """Plant one of the FAULT_* mistakes (negative-control tests only)."""
    _load().oracle_set_fault(int(f))


class scale_rule:
    """Context manager: run the quantizers under a scale rule (UE8M0 scales,
    amax floor, scale floor); the default rule is restored on exit."""

    def __init__(self, ue8m0: bool = False, amax_floor: float = 0.0, scale_floor: float = 0.0):
        self.args = (int(bool(ue8m0)), float(amax_floor), float(scale_floor))

    def __enter__(self):
        _load().oracle_set_scale_rule(*self.args)
        return self

    def __exit__(self, *exc):
        _load().oracle_set_scale_rule(0, 0.0, 0.0)
        return False


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


# ---------------------------------------------------------------------------
# E4M3 and bf16 helpers
# ---------------------------------------------------------------------------

def e4m3_table() -> np.ndarray:
    """float32[256]: the value of every E4M3 code (NaN for 0x7F and 0xFF)."""
    out = np.empty(256, np.float32)
    _load().oracle_e4m3_table(_p(out))
    return out


def e4m3_encode(v: float) -> int:
    return int(_load().oracle_e4m3_encode(float(v)))


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    flat = _c(np.asarray(v, np.float32).ravel(), np.float32)
    out = np.empty(flat.size, np.uint8)
    _load().oracle_e4m3_encode_array(_p(flat), flat.size, _p(out))
    return out.reshape(np.shape(v))


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return e4m3_table()[np.asarray(codes, np.uint8)]


def f32_to_bf16(v: np.ndarray) -> np.ndarray:
    v = _c(v, np.float32)
    out = np.empty(v.shape, np.uint16)
    _load().oracle_f32_to_bf16_array(_p(v), v.size, _p(out))
    return out


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Quantizers
# ---------------------------------------------------------------------------

def scale_rows_padded(rows: int) -> int:
    """Row count of the 1x128 scale array (rows rounded up to a multiple of 4)."""
    return (rows + 3) // 4 * 4


def quant_1x128(x_bf16: np.ndarray, sc_layout: str = "tile_major"):
    """1x128 tiles along each row of x [R x C].

    Returns (q uint8 [R x C], scales). ``tile_major`` gives scales as
    float32 [ceil(C/128) x pad4(R)] (row index contiguous, padding zero);
    ``row_major`` gives float32 [R x ceil(C/128)].
    """
    x = _c(x_bf16, np.uint16)
    R, C = x.shape
    nt = (C + 127) // 128
    q = np.empty((R, C), np.uint8)
    if sc_layout == "tile_major":
        rp = scale_rows_padded(R)
        sc = np.zeros((nt, rp), np.float32)
        rs, ts = 1, rp
    else:
        sc = np.zeros((R, nt), np.float32)
        rs, ts = nt, 1
    _load().oracle_quant_1x128(_p(x), R, C, C, _p(q), C, _p(sc), rs, ts)
    return q, sc


def quant_128x128(w_bf16: np.ndarray):
    """128x128 blocks of w [R x C]. Returns (q uint8 [R x C], scales
    float32 [ceil(R/128) x ceil(C/128)])."""
    w = _c(w_bf16, np.uint16)
    R, C = w.shape
    q = np.empty((R, C), np.uint8)
    sc = np.zeros(((R + 127) // 128, (C + 127) // 128), np.float32)
    _load().oracle_quant_128x128(_p(w), R, C, C, _p(q), C, _p(sc), sc.shape[1])
    return q, sc


def philox4x32_10(counter, key):
    """Philox4x32-10 of a 4-word counter and 2-word key -> 4 words."""
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    _load().oracle_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def sr_word(seed: int, salt: int, idx: int) -> int:
    return int(_load().oracle_sr_word(int(seed), int(salt), int(idx)))


def e4m3_encode_sr(x: float, r: int) -> int:
    return int(_load().oracle_e4m3_encode_sr(float(x), int(r)))


def quant_1x128_sr(x_bf16: np.ndarray, seed: int, salt: int = 0):
    """quant_1x128 with stochastic rounding (tile-major scales)."""
    x = _c(x_bf16, np.uint16)
    R, C = x.shape
    nt = (C + 127) // 128
    q = np.empty((R, C), np.uint8)
    rp = scale_rows_padded(R)
    sc = np.zeros((nt, rp), np.float32)
    _load().oracle_quant_1x128_sr(_p(x), R, C, C, _p(q), C, _p(sc), 1, rp, int(seed), int(salt))
    return q, sc


def quant_128x128_sr(w_bf16: np.ndarray, seed: int, salt: int = 0, idx_base: int = 0):
    """quant_128x128 with stochastic rounding; element indices start at idx_base."""
    w = _c(w_bf16, np.uint16)
    R, C = w.shape
    q = np.empty((R, C), np.uint8)
    sc = np.zeros(((R + 127) // 128, (C + 127) // 128), np.float32)
    _load().oracle_quant_128x128_sr(_p(w), R, C, C, _p(q), C, _p(sc), sc.shape[1], int(seed), int(salt),
                                    int(idx_base))
    return q, sc


def mx_quant_1x32(x_bf16: np.ndarray):
    """MXFP8 1x32 blocks along the rows of x [R x C] (C % 32 == 0).
    Returns (q uint8 [R x C], exponent bytes uint8 [R x C/32])."""
    x = _c(x_bf16, np.uint16)
    R, C = x.shape
    assert C % 32 == 0
    q = np.empty((R, C), np.uint8)
    sc = np.empty((R, C // 32), np.uint8)
    _load().oracle_mx_quant_1x32(_p(x), R, C, _p(q), _p(sc))
    return q, sc


def mx_gemm(a, sa, b, sb, ii=None, jj=None):
    """MXFP8 GEMM of A [M x K] and B [N x K] (both 1x32-blocked along K):
    fp32 [M x N] (or the sampled elements)."""
    a, b = _c(a, np.uint8), _c(b, np.uint8)
    sa, sb = _c(sa, np.uint8), _c(sb, np.uint8)
    M, K = a.shape
    N = b.shape[0]
    if ii is None:
        out = np.empty((M, N), np.float32)
        _load().oracle_mx_gemm(_p(a), _p(sa), _p(b), _p(sb), M, N, K, _p(out), None, None, 0)
    else:
        ii, jj = _c(ii, np.int64), _c(jj, np.int64)
        out = np.empty(ii.size, np.float32)
        _load().oracle_mx_gemm(_p(a), _p(sa), _p(b), _p(sb), M, N, K, _p(out), _p(ii), _p(jj), ii.size)
    return out


def pack_ue8m0(scales, rows: int, K: int, row_block: int, row_stride: int, kb_stride: int):
    """Exponent bytes of power-of-two block scales for the MX GEMM, in the
    plain layout [rows x K/32] (one byte per row and 32-element block of K).

    Follows the "Compact formats" row of the prime-rl conventions table
    (Blackwell consumes the scales as packed exponent bytes) read with the
    OCP MX v1.0 exponent-byte format: s = 2^(E - 127), E in 0..254, 255 = NaN.
    The scale of (row r, 128-element K-block b) is
    scales.ravel()[(r // row_block) * row_stride + b * kb_stride]; each
    K-block's byte covers its four 32-element blocks. A scale that is not an
    exact positive power of two in [2^-127, 2^127] has no byte: 255.
    Returns (bytes uint8 [rows x K/32], count of scales without a byte).
    """
    flat = np.asarray(scales, np.float32).ravel()
    kb = K // 128
    r = np.arange(rows, dtype=np.int64)[:, None]
    b = np.arange(kb, dtype=np.int64)[None, :]
    s = flat[(r // row_block) * row_stride + b * kb_stride].astype(np.float64)   # [rows x kb]
    with np.errstate(invalid="ignore"):
        m, e = np.frexp(s)                  # s = m * 2^e with m in [0.5, 1) for finite s > 0
        E = e.astype(np.int64) + 126        # s = 2^(e - 1) = 2^(E - 127) exactly when m == 0.5
        ok = (m == 0.5) & (E >= 0) & (E <= 254)
    byte = np.where(ok, E, 255).astype(np.uint8)
    return np.repeat(byte, 4, axis=1), int(np.count_nonzero(~ok))


def padded_tokens(rows: int, offsets=None) -> int:
    if offsets is None:
        return (rows + 127) // 128 * 128
    off = _c(offsets, np.int32)
    return int(_load().oracle_padded_tokens(_p(off), off.size - 1, rows))


def requant_128x1_T(src: np.ndarray, src_scales: np.ndarray | None = None, offsets=None, sr=None):
    """128x1 (token-axis) tiles of src [M x C], transposed output.

    src is bf16 bits (uint16, mode B) or E4M3 codes (uint8, mode Q, with its
    1x128 scales in the tile-major layout of ``quant_1x128``). ``offsets``
    (int32, G+1 entries) splits the rows into groups whose tiles start at
    their own first row. Returns (qT uint8 [C x Mpad], scT float32
    [Mpad/128 x C]) where each group's segment is padded to 128 tokens.
    """
    src = np.ascontiguousarray(src)
    M, C = src.shape
    mode = 0 if src.dtype == np.uint16 else 1
    if mode == 1:
        assert src.dtype == np.uint8 and src_scales is not None
        ssc = _c(src_scales, np.float32)
        rs, ts = 1, ssc.shape[1]
    else:
        ssc, rs, ts = None, 0, 0
    if offsets is not None:
        off = _c(offsets, np.int32)
        G = off.size - 1
        assert off[0] == 0 and off[-1] == M
    else:
        off, G = None, 0
    mp = padded_tokens(M, off)
    qT = np.zeros((C, mp), np.uint8)
    scT = np.zeros((mp // 128, C), np.float32)
    if sr is None:
        _load().oracle_requant_128x1_T(mode, _p(src), C, _p(ssc), rs, ts, M, C,
                                       _p(off), G, _p(qT), mp, _p(scT), C)
    else:
        _load().oracle_requant_128x1_T_sr(mode, _p(src), C, _p(ssc), rs, ts, M, C,
                                          _p(off), G, _p(qT), mp, _p(scT), C, int(sr[0]), int(sr[1]))
    return qT, scT


def requant_128x1_T_sr(src: np.ndarray, src_scales: np.ndarray | None = None, offsets=None, *,
                       seed: int, salt: int = 0):
    """requant_128x1_T with stochastic rounding: source element (r, c) takes
    the random word of index r * C + c under (seed, salt)."""
    return requant_128x1_T(src, src_scales, offsets, sr=(seed, salt))


# ---------------------------------------------------------------------------
# Promoted GEMMs. Outputs are fp32 values before the BF16 rounding of Y / dX
# (use f32_to_bf16 for that); dW is fp32 by definition.
# ---------------------------------------------------------------------------

def _idx(ii, jj):
    if ii is None:
        return None, None, 0
    ii = _c(ii, np.int64)
    jj = _c(jj, np.int64)
    assert ii.shape == jj.shape
    return ii, jj, ii.size


def fprop(xq, sx, wq, sw, ii=None, jj=None):
    """Y = X W. xq uint8 [M x K]; sx tile-major [K/128 x pad4(M)];
    wq uint8 [K x N]; sw [K/128 x N/128]. Full [M x N] fp32, or the listed
    elements (ii, jj)."""
    xq = _c(xq, np.uint8); wq = _c(wq, np.uint8)
    sx = _c(sx, np.float32); sw = _c(sw, np.float32)
    M, K = xq.shape
    K2, N = wq.shape
    assert K == K2
    ii, jj, n = _idx(ii, jj)
    out = np.empty(n if ii is not None else (M, N), np.float32)
    _load().oracle_fprop(_p(xq), K, _p(sx), 1, sx.shape[1], _p(wq), N, _p(sw), sw.shape[1],
                         M, N, K, _p(ii), _p(jj), n, _p(out))
    return out


def dgrad(dyq, sdy, wq, sw, ii=None, kk=None):
    """dX = dY W^T. dyq uint8 [M x N]; sdy tile-major [N/128 x pad4(M)];
    wq uint8 [K x N]; sw [K/128 x N/128]. Full [M x K] fp32 or listed."""
    dyq = _c(dyq, np.uint8); wq = _c(wq, np.uint8)
    sdy = _c(sdy, np.float32); sw = _c(sw, np.float32)
    M, N = dyq.shape
    K, N2 = wq.shape
    assert N == N2
    ii, kk, n = _idx(ii, kk)
    out = np.empty(n if ii is not None else (M, K), np.float32)
    _load().oracle_dgrad(_p(dyq), N, _p(sdy), 1, sdy.shape[1], _p(wq), N, _p(sw), sw.shape[1],
                         M, N, K, _p(ii), _p(kk), n, _p(out))
    return out


def wgrad(dyqT, sdyT, xqT, sxT, nn=None, kk=None, t0=0, t1=None):
    """dW = dY^T X on the transposed 128x1 operands. dyqT uint8 [N x T];
    sdyT [T/128 x N]; xqT uint8 [K x T]; sxT [T/128 x K]. The contraction
    runs over padded tokens [t0, t1) (whole 128-token tiles). Full [N x K]
    fp32 or the listed elements."""
    dyqT = _c(dyqT, np.uint8); xqT = _c(xqT, np.uint8)
    sdyT = _c(sdyT, np.float32); sxT = _c(sxT, np.float32)
    N, T = dyqT.shape
    K, T2 = xqT.shape
    assert T == T2
    if t1 is None:
        t1 = T
    assert t0 % 128 == 0 and t1 % 128 == 0 and 0 <= t0 <= t1 <= T
    nn, kk, n = _idx(nn, kk)
    out = np.empty(n if nn is not None else (N, K), np.float32)
    if t1 == t0:
        out[...] = 0.0
        return out
    b0 = t0 // 128
    a_ptr = ctypes.c_void_p(dyqT.ctypes.data + t0)
    b_ptr = ctypes.c_void_p(xqT.ctypes.data + t0)
    sa_ptr = ctypes.c_void_p(sdyT.ctypes.data + b0 * N * 4)
    sb_ptr = ctypes.c_void_p(sxT.ctypes.data + b0 * K * 4)
    _load().oracle_wgrad(a_ptr, T, sa_ptr, N, b_ptr, T, sb_ptr, K,
                         t1 - t0, N, K, _p(nn), _p(kk), n, _p(out))
    return out


def fprop_reference_sums(xq, sx, wq, sw, ii, jj, m_bits=14, mode=0, unpromoted=True):
    """For listed elements of Y = X W: (fp64 sum over dequantized operands,
    unpromoted m-bit accumulation of the drift model or None)."""
    xq = _c(xq, np.uint8); wq = _c(wq, np.uint8)
    sx = _c(sx, np.float32); sw = _c(sw, np.float32)
    M, K = xq.shape
    _, N = wq.shape
    ii, jj, n = _idx(ii, jj)
    t = np.empty(n, np.float64)
    u = np.empty(n, np.float64) if unpromoted else None
    _load().oracle_fprop_reference_sums(_p(xq), K, _p(sx), 1, sx.shape[1], _p(wq), N,
                                        _p(sw), sw.shape[1], K, _p(ii), _p(jj), n,
                                        int(m_bits), int(mode), _p(t), _p(u))
    return t, u


def round_sig(v: float, m: int, mode: int = 0) -> float:
    return float(_load().oracle_round_sig(float(v), int(m), int(mode)))


# ---------------------------------------------------------------------------
# Grouped (MoE) variants: the dense definitions applied to each expert.
# ---------------------------------------------------------------------------

def grouped_fprop(xq, sx, wq_stack, sw_stack, offsets):
    """Per expert e: Y[rows of e] = X[rows of e] W_e. Full fp32 [M x N]."""
    M = xq.shape[0]
    N = wq_stack.shape[2]
    out = np.zeros((M, N), np.float32)
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        # the 1x128 scales of rows r0..r1 are columns r0..r1 of the tile-major array
        out[r0:r1] = fprop(xq[r0:r1], np.ascontiguousarray(sx[:, r0:r1]), wq_stack[e],
                           sw_stack[e])
    return out
