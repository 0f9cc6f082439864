"""Shared helpers for the parity tests: the GEMM tolerance and small
marshalling utilities between torch tensors and the oracle's numpy arrays.

Tolerance (stated for the GEMMs, per output element, over the dequantized
operands a_k, b_k of that element):
    |gpu - oracle| <= 2e-3 * sum_k |a_k b_k| + 1e-6     (+ one BF16 ulp of
                                                       |oracle| for BF16 outputs)
The quantizers are compared bit for bit (payload bytes and fp32 scale bits).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

REL_TOL = 2e-3
ABS_TOL = 1e-6


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def np_(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy()


def bf16_values(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def bf16_ulp(y: np.ndarray) -> np.ndarray:
    a = np.abs(y.astype(np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -133)))
    return np.exp2(e - 7)


def dequant_rows(q: np.ndarray, sc_tile_major: np.ndarray, rows=None) -> np.ndarray:
    """Dequantize rows of a 1x128-quantized [R x C] payload (fp64)."""
    t = oracle.e4m3_table().astype(np.float64)
    if rows is None:
        rows = np.arange(q.shape[0])
    C = q.shape[1]
    s = sc_tile_major[:, rows].T.astype(np.float64)          # [len(rows) x C/128]
    return t[q[rows]] * np.repeat(s, 128, axis=1)[:, :C]


def dequant_blocks(q: np.ndarray, sc: np.ndarray) -> np.ndarray:
    t = oracle.e4m3_table().astype(np.float64)
    s = np.repeat(np.repeat(sc.astype(np.float64), 128, 0), 128, 1)[:q.shape[0], :q.shape[1]]
    return t[q] * s


def dequant_tokens_T(qT: np.ndarray, scT: np.ndarray) -> np.ndarray:
    """Dequantize a transposed 128x1 payload [C x T] with scales [T/128 x C]."""
    t = oracle.e4m3_table().astype(np.float64)
    return t[qT] * np.repeat(scT.T.astype(np.float64), 128, axis=1)


def assert_gemm_close(gpu: np.ndarray, ref: np.ndarray, absprod: np.ndarray, bf16_out: bool,
                      what: str = "") -> None:
    gpu = gpu.astype(np.float64)
    ref = ref.astype(np.float64)
    tol = REL_TOL * absprod + ABS_TOL
    if bf16_out:
        tol = tol + bf16_ulp(ref)
    err = np.abs(gpu - ref)
    bad = err > tol
    if bad.any():
        i = np.argmax(err - tol)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; worst at flat "
            f"index {i}: gpu={gpu.flat[i]!r} oracle={ref.flat[i]!r} tol={tol.flat[i]!r}")


def sample_indices(M: int, N: int, n: int, seed: int, tiles=((0, 0),), tile=128):
    """Seeded random output coordinates plus every element of the listed
    128x128 output tiles (negative tile indices count from the end)."""
    g = np.random.default_rng(seed)
    ii = [g.integers(0, M, n)]
    jj = [g.integers(0, N, n)]
    for (ti, tj) in tiles:
        ti = ti % ((M + tile - 1) // tile)
        tj = tj % ((N + tile - 1) // tile)
        r = np.arange(ti * tile, min(M, ti * tile + tile))
        c = np.arange(tj * tile, min(N, tj * tile + tile))
        rr, cc = np.meshgrid(r, c, indexing="ij")
        ii.append(rr.ravel())
        jj.append(cc.ravel())
    return np.concatenate(ii).astype(np.int64), np.concatenate(jj).astype(np.int64)


def absprod_sampled(a_abs: np.ndarray, bt_abs: np.ndarray, ii: np.ndarray, jj: np.ndarray,
                    chunk: int = 2048) -> np.ndarray:
    """sum_k a_abs[ii[e], k] * bt_abs[jj[e], k] for each sampled element e,
    in chunks (a_abs: [rows x K], bt_abs: [cols x K])."""
    out = np.empty(ii.size, np.float64)
    for s in range(0, ii.size, chunk):
        out[s:s + chunk] = np.einsum("ek,ek->e", a_abs[ii[s:s + chunk]], bt_abs[jj[s:s + chunk]])
    return out
