"""GB300 (sm_103a) fine-grained FP8 linear layer: Python binding of libfp8bs.

Thin ctypes binding of the C ABI declared in ``include/fp8bs.h``. Each function
has the name of its C entry point and only marshals arguments: torch tensors
supply device pointers and sizes, the current torch CUDA stream supplies the
stream, and every step of the computation runs in the library's CUDA
kernels. There is no fallback: if ``libfp8bs.so`` is missing or fails to load,
every call raises.

PyTorch is used here for device memory and streams only. Allocation helpers
(``empty_*``) return correctly shaped output tensors for each entry point.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch

from . import _build_lib

__all__ = [
    "Fp8bsError", "build", "lib", "lib_path",
    "fp8_quant_1x128", "fp8_quant_128x128", "fp8_requant_128x1_T", "fp8_quant_dual",
    "fp8_block_gemm_fprop", "fp8_block_gemm_fprop_wkn", "fp8_block_gemm_dgrad", "fp8_block_gemm_wgrad",
    "fp8_block_gemm_grouped", "fp8_block_gemm_splitk", "fp8bs_splitk_workspace_size",
    "fp8bs_splitk_default_splits", "fp8_block_gemm_splitk_noalloc", "NOALLOC_SCRATCH_BYTES",
    "fp8bs_device_status", "fp8bs_last_device_status", "fp8bs_copy_device_status", "fp8bs_set_wait_limit_ns",
    "fp8bs_padded_tokens_max", "fp8_requant_128x1_T_dev", "fp8_quant_dual_dev", "fp8_quant_dual_stash_dev",
    "fp8bs_selftest_wait_timeout", "fp8bs_selftest_gemm_timeout", "fp8bs_scale_ld", "fp8bs_padded_tokens",
    "fp8bs_status_str", "fp8bs_version",
    "empty_quant_1x128", "empty_quant_128x128", "empty_requant_128x1_T",
    "SRC_BF16", "SRC_E4M3", "OP_FPROP", "OP_DGRAD", "OP_WGRAD", "OP_FPROP_WKN", "MAX_GROUPS",
    "SCALE_FP32", "SCALE_UE8M0", "ScaleOpts", "fp8_quant_1x128_opts", "fp8_quant_128x128_opts",
    "fp8_requant_128x1_T_opts", "fp8_quant_dual_opts", "fp8_quant_1x128_sr", "fp8_quant_128x128_sr",
    "fp8_quant_dual_stash", "fp8_quant_dual_stash_opts", "fp8_requant_128x1_T_sr", "fp8_quant_dual_sr",
    "fp8_quant_dual_stash_sr",
    "fp8bs_mx_scale_bytes", "fp8_mx_quant_1x32", "fp8_mx_gemm", "empty_mx_quant",
    "fp8_mx_quant_1x32_T", "fp8_mx_gemm_f32", "fp8_mx_gemm_wkn", "empty_mx_quant_T", "fp8_pack_ue8m0",
    "fp8_mx_gemm_grouped", "fp8_pack_ue8m0_grouped",
    "fp8_quant_128x128_packed", "fp8_quant_dual_packed", "fp8_quant_dual_stash_packed", "empty_mx_atoms",
    "fp8_quant_dual_packed_grouped", "fp8_quant_dual_stash_packed_grouped",
]

SRC_BF16, SRC_E4M3 = 0, 1
SCALE_FP32, SCALE_UE8M0 = 0, 1
OP_FPROP, OP_DGRAD, OP_WGRAD, OP_FPROP_WKN = 0, 1, 2, 3
MAX_GROUPS = 256
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024   # FP8BS_NOALLOC_SCRATCH_BYTES
STATUS_NAMES = {0: "OK", 1: "ERR_ARG", 2: "ERR_ALIGN", 3: "ERR_SHAPE", 4: "ERR_LAUNCH",
                5: "ERR_TIMEOUT", 6: "ERR_UNSUPPORTED", 7: "ERR_DEVICE"}

_lib = None


class ScaleOpts(ctypes.Structure):
    """fp8bs_scale_opts: the quantizers' scale rule (see fp8bs.h)."""
    _fields_ = [("rule", ctypes.c_int32), ("amax_floor", ctypes.c_float), ("scale_floor", ctypes.c_float)]


class Fp8bsError(RuntimeError):
    def __init__(self, fn: str, code: int, detail: str = ""):
        self.code = int(code)
        msg = f"{fn}: {STATUS_NAMES.get(self.code, self.code)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))


def lib_path() -> str:
    return _build_lib.LIB


def build(force: bool = False) -> str:
    """Compile libfp8bs.so for sm_103a (nvcc) if its sources changed."""
    return _build_lib.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded C library. Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libfp8bs.so not found at {path}: run "
                           "fp8_block_scaled_act_gb300.build() (nvcc, sm_103a) first")
    L = ctypes.CDLL(path)
    P, I64, I32, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
    S = ctypes.c_int
    sigs = {
        "fp8bs_status_str": ([S], ctypes.c_char_p),
        "fp8bs_version": ([], I),
        "fp8bs_scale_ld": ([I64], I64),
        "fp8bs_padded_tokens": ([I64, P, I32], I64),
        "fp8_quant_1x128": ([P, I64, I64, I64, P, P, P], S),
        "fp8_quant_128x128": ([P, I64, I64, I64, I64, P, P, P, P], S),
        "fp8_requant_128x1_T": ([I, P, P, I64, I64, P, I32, P, P, P], S),
        "fp8_quant_dual": ([P, I64, I64, P, I32, P, P, P, P, P], S),
        "fp8_quant_1x128_opts": ([P, I64, I64, I64, P, P, P, P], S),
        "fp8_quant_128x128_opts": ([P, I64, I64, I64, I64, P, P, P, P, P], S),
        "fp8_requant_128x1_T_opts": ([I, P, P, I64, I64, P, I32, P, P, P, P], S),
        "fp8_quant_dual_opts": ([P, I64, I64, P, I32, P, P, P, P, P, P], S),
        "fp8_quant_dual_stash": ([P, I64, I64, P, I32, P, P, P, P, P], S),
        "fp8_quant_dual_stash_opts": ([P, I64, I64, P, I32, P, P, P, P, P, P], S),
        "fp8_quant_1x128_sr": ([P, I64, I64, I64, P, P, ctypes.c_uint64, ctypes.c_uint32, P, P], S),
        "fp8_requant_128x1_T_sr": ([I, P, P, I64, I64, P, I32, P, P, ctypes.c_uint64, ctypes.c_uint32, P, P], S),
        "fp8_quant_dual_sr": ([P, I64, I64, P, I32, P, P, P, P, ctypes.c_uint64, ctypes.c_uint32, P, P], S),
        "fp8_quant_dual_stash_sr": ([P, I64, I64, P, I32, P, P, P, P, ctypes.c_uint64, ctypes.c_uint32, P, P], S),
        "fp8bs_mx_scale_bytes": ([I64, I64], I64),
        "fp8_mx_quant_1x32": ([P, I64, I64, P, P, P], S),
        "fp8_mx_gemm": ([P, P, P, P, I64, I64, I64, P, P], S),
        "fp8_mx_gemm_wkn": ([P, P, P, P, I64, I64, I64, P, P], S),
        "fp8_mx_gemm_f32": ([P, P, P, P, I64, I64, I64, P, P], S),
        "fp8_mx_gemm_grouped": ([I, I32, P, P, I64, P, P, P, P, I64, I64, P, P], S),
        "fp8_pack_ue8m0_grouped": ([P, I64, I64, I64, I32, P, P, P, P], S),
        "fp8_mx_quant_1x32_T": ([P, I64, I64, P, P, P], S),
        "fp8_pack_ue8m0": ([P, I64, I64, I32, I64, I64, P, P], S),
        "fp8_quant_128x128_packed": ([P, I64, I64, I64, I64, P, P, P, P, P, P, P], S),
        "fp8_quant_dual_packed": ([P, I64, I64, P, P, P, P, P, P, P, P], S),
        "fp8_quant_dual_stash_packed": ([P, I64, I64, P, P, P, P, P, P, P, P], S),
        "fp8_quant_dual_packed_grouped": ([P, I64, I64, P, P, I32, P, P, P, P, P, P, P, P], S),
        "fp8_quant_dual_stash_packed_grouped": ([P, I64, I64, P, P, I32, P, P, P, P, P, P, P, P], S),
        "fp8_quant_128x128_sr": ([P, I64, I64, I64, I64, P, P, P, ctypes.c_uint64, ctypes.c_uint32, P, P], S),
        "fp8_block_gemm_fprop": ([P, P, P, P, I64, I64, I64, P, P], S),
        "fp8_block_gemm_fprop_wkn": ([P, P, P, P, I64, I64, I64, P, P], S),
        "fp8_block_gemm_dgrad": ([P, P, P, P, I64, I64, I64, P, P], S),
        "fp8_block_gemm_wgrad": ([P, P, P, P, I64, I64, I64, P, I, P], S),
        "fp8_block_gemm_grouped": ([I, I32, P, P, I64, P, P, P, P, I64, I64, P, I, P], S),
        "fp8bs_padded_tokens_max": ([I64, I32], I64),
        "fp8_requant_128x1_T_dev": ([I, P, P, I64, I64, P, I32, P, P, P, P], S),
        "fp8_quant_dual_dev": ([P, I64, I64, P, I32, P, P, P, P, P, P], S),
        "fp8_quant_dual_stash_dev": ([P, I64, I64, P, I32, P, P, P, P, P, P], S),
        "fp8bs_last_device_status": ([P, I], S),
        "fp8bs_copy_device_status": ([P, I, P], S),
        "fp8bs_splitk_workspace_size": ([I, I64, I64, I64, I32], ctypes.c_size_t),
        "fp8bs_splitk_default_splits": ([I, I64, I64, I64], I32),
        "fp8_block_gemm_splitk": ([I, P, P, P, P, I64, I64, I64, I32, P, P, ctypes.c_size_t, P], S),
        "fp8_block_gemm_splitk_noalloc": ([I, P, P, P, P, I64, I64, I64, I32, P, P], S),
        "fp8bs_device_status": ([I], S),
        "fp8bs_set_wait_limit_ns": ([ctypes.c_uint64], None),
        "fp8bs_selftest_wait_timeout": ([ctypes.c_uint64, P], S),
        "fp8bs_selftest_gemm_timeout": ([P, P, P, P, I64, I64, I64, P, ctypes.c_uint64, P], S),
    }
    for name, (args, res) in sigs.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _opts(rule: int, amax_floor: float, scale_floor: float):
    """ctypes pointer to a ScaleOpts, or None for the default rule."""
    if rule == SCALE_FP32 and amax_floor == 0.0 and scale_floor == 0.0:
        return None
    return ctypes.pointer(ScaleOpts(int(rule), float(amax_floor), float(scale_floor)))


def _check(name: str, code: int, detail: str = "") -> None:
    if code != 0:
        raise Fp8bsError(name, code, detail)


def _need(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _on_device(offsets) -> bool:
    """Group offsets given as a CUDA tensor are read by the kernels on the
    device (the _dev entry points); anything else is a host array."""
    return isinstance(offsets, torch.Tensor) and offsets.is_cuda


def _offsets_dev(offsets: torch.Tensor):
    _need(offsets, torch.int32, "offsets")
    if offsets.dim() != 1 or offsets.numel() < 2:
        raise ValueError("offsets: 1-D int32 tensor of groups + 1 entries")
    return _ptr(offsets), offsets.numel() - 1


def _offsets_host(offsets) -> np.ndarray:
    if isinstance(offsets, torch.Tensor):
        offsets = offsets.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(offsets, dtype=np.int32))


# ---------------------------------------------------------------------------
# helpers without device work
# ---------------------------------------------------------------------------

def fp8bs_status_str(code: int) -> str:
    return lib().fp8bs_status_str(int(code)).decode()


def fp8bs_version() -> int:
    return int(lib().fp8bs_version())


def fp8bs_scale_ld(rows: int) -> int:
    return int(lib().fp8bs_scale_ld(int(rows)))


def fp8bs_padded_tokens(rows: int, offsets: Optional[Sequence[int]] = None) -> int:
    if offsets is None:
        return int(lib().fp8bs_padded_tokens(int(rows), None, 0))
    off = _offsets_host(offsets)
    v = int(lib().fp8bs_padded_tokens(int(rows), off.ctypes.data_as(ctypes.c_void_p), off.size - 1))
    if v < 0:
        raise ValueError("invalid group offsets")
    return v


def empty_quant_1x128(rows: int, cols: int, device="cuda"):
    """(q uint8 [rows x cols], scales float32 [ceil(cols/128) x scale_ld(rows)])."""
    q = torch.empty((rows, cols), dtype=torch.uint8, device=device)
    sc = torch.empty(((cols + 127) // 128, max(fp8bs_scale_ld(rows), 0)), dtype=torch.float32,
                     device=device)
    return q, sc


def empty_quant_128x128(rows: int, cols: int, batch: Optional[int] = None,
                        with_transpose: bool = True, device="cuda"):
    """(q [batch x rows x cols], qT [batch x cols x rows] or None, scales
    [batch x ceil(rows/128) x ceil(cols/128)]); without ``batch`` the tensors
    have no batch dimension."""
    shp = (int(batch),) if batch is not None else ()
    q = torch.empty(shp + (rows, cols), dtype=torch.uint8, device=device)
    qT = torch.empty(shp + (cols, rows), dtype=torch.uint8, device=device) if with_transpose else None
    sc = torch.empty(shp + ((rows + 127) // 128, (cols + 127) // 128), dtype=torch.float32,
                     device=device)
    return q, qT, sc


def fp8bs_padded_tokens_max(rows: int, groups: int) -> int:
    v = int(lib().fp8bs_padded_tokens_max(int(rows), int(groups)))
    if v < 0:
        raise ValueError("invalid rows or groups")
    return v


def _padded(rows: int, offsets) -> int:
    """Token length of the transposed outputs: exact for host offsets, the
    capacity bound for device offsets."""
    if _on_device(offsets):
        return fp8bs_padded_tokens_max(rows, offsets.numel() - 1)
    return fp8bs_padded_tokens(rows, offsets)


def empty_requant_128x1_T(rows: int, cols: int, offsets=None, device="cuda"):
    """(qT uint8 [cols x Mpad], scalesT float32 [Mpad/128 x cols]); with
    device offsets Mpad is fp8bs_padded_tokens_max(rows, groups)."""
    mp = _padded(rows, offsets)
    qT = torch.empty((cols, mp), dtype=torch.uint8, device=device)
    sc = torch.empty((mp // 128, cols), dtype=torch.float32, device=device)
    return qT, sc


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def fp8_quant_1x128(x: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, stream=None,
                    rule: int = SCALE_FP32, amax_floor: float = 0.0, scale_floor: float = 0.0) -> None:
    """1x128 absmax quantization of BF16 x [rows x cols] into q / scales
    (optional scale rule: UE8M0 rounding, amax / scale floors)."""
    _need(x, torch.bfloat16, "x"); _need(q, torch.uint8, "q"); _need(scales, torch.float32, "scales")
    rows, cols = x.shape
    if q.shape != (rows, cols) or scales.shape != ((cols + 127) // 128, fp8bs_scale_ld(rows)):
        raise ValueError("output shapes do not match empty_quant_1x128")
    _check("fp8_quant_1x128", lib().fp8_quant_1x128_opts(_ptr(x), rows, cols, cols, _ptr(q), _ptr(scales),
                                                         _opts(rule, amax_floor, scale_floor), _stream(stream)))


def fp8_quant_128x128(w: torch.Tensor, q: torch.Tensor, qT: Optional[torch.Tensor],
                      scales: torch.Tensor, stream=None, rule: int = SCALE_FP32, amax_floor: float = 0.0,
                      scale_floor: float = 0.0) -> None:
    """128x128 absmax quantization of BF16 w [rows x cols] (or [batch x rows x cols])."""
    _need(w, torch.bfloat16, "w"); _need(q, torch.uint8, "q"); _need(scales, torch.float32, "scales")
    if qT is not None:
        _need(qT, torch.uint8, "qT")
    batch = w.shape[0] if w.dim() == 3 else 1
    rows, cols = w.shape[-2:]
    nb = ((rows + 127) // 128) * ((cols + 127) // 128)
    if (q.numel() != w.numel() or q.shape[-2:] != (rows, cols) or scales.numel() != batch * nb
            or (qT is not None and (qT.numel() != w.numel() or qT.shape[-2:] != (cols, rows)))):
        raise ValueError("output shapes do not match empty_quant_128x128")
    _check("fp8_quant_128x128", lib().fp8_quant_128x128_opts(_ptr(w), batch, rows, cols, cols, _ptr(q),
                                                             _ptr(qT), _ptr(scales),
                                                             _opts(rule, amax_floor, scale_floor), _stream(stream)))


def fp8_requant_128x1_T_sr(src: torch.Tensor, src_scales: Optional[torch.Tensor], qT: torch.Tensor,
                           scalesT: torch.Tensor, seed: int, salt: int = 0, offsets=None, stream=None,
                           rule: int = SCALE_FP32, amax_floor: float = 0.0, scale_floor: float = 0.0) -> None:
    """fp8_requant_128x1_T with stochastic rounding under (seed, salt); see fp8bs.h."""
    fp8_requant_128x1_T(src, src_scales, qT, scalesT, offsets, stream, rule, amax_floor, scale_floor,
                        sr=(seed, salt))


def fp8_requant_128x1_T(src: torch.Tensor, src_scales: Optional[torch.Tensor], qT: torch.Tensor,
                        scalesT: torch.Tensor, offsets=None, stream=None, rule: int = SCALE_FP32,
                        amax_floor: float = 0.0, scale_floor: float = 0.0, sr=None) -> None:
    """128x1 transposed requantization. src BF16 (mode B) or uint8 E4M3 with
    its 1x128 scales (mode Q); optional host group offsets; sr = (seed, salt)
    selects stochastic rounding."""
    if src.dtype == torch.bfloat16:
        mode = SRC_BF16
        _need(src, torch.bfloat16, "src")
    else:
        mode = SRC_E4M3
        _need(src, torch.uint8, "src"); _need(src_scales, torch.float32, "src_scales")
    _need(qT, torch.uint8, "qT"); _need(scalesT, torch.float32, "scalesT")
    rows, cols = src.shape
    mp = _padded(rows, offsets)
    if qT.shape != (cols, mp) or scalesT.shape != (mp // 128, cols):
        raise ValueError("output shapes do not match empty_requant_128x1_T")
    if _on_device(offsets):
        if sr is not None:
            raise ValueError("stochastic rounding takes host offsets")
        optr, groups = _offsets_dev(offsets)
        _check("fp8_requant_128x1_T_dev", lib().fp8_requant_128x1_T_dev(
            mode, _ptr(src), _ptr(src_scales if mode == SRC_E4M3 else None), rows, cols, optr, groups,
            _ptr(qT), _ptr(scalesT), _opts(rule, amax_floor, scale_floor), _stream(stream)))
        return
    if offsets is not None:
        off = _offsets_host(offsets)
        optr, groups = off.ctypes.data_as(ctypes.c_void_p), off.size - 1
    else:
        off, optr, groups = None, None, 0
    if sr is None:
        _check("fp8_requant_128x1_T", lib().fp8_requant_128x1_T_opts(
            mode, _ptr(src), _ptr(src_scales if mode == SRC_E4M3 else None), rows, cols, optr, groups,
            _ptr(qT), _ptr(scalesT), _opts(rule, amax_floor, scale_floor), _stream(stream)))
    else:
        _check("fp8_requant_128x1_T_sr", lib().fp8_requant_128x1_T_sr(
            mode, _ptr(src), _ptr(src_scales if mode == SRC_E4M3 else None), rows, cols, optr, groups,
            _ptr(qT), _ptr(scalesT), int(sr[0]) & (2 ** 64 - 1), int(sr[1]) & 0xFFFFFFFF,
            _opts(rule, amax_floor, scale_floor), _stream(stream)))


def fp8_quant_dual(x: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, qT: torch.Tensor,
                   scalesT: torch.Tensor, offsets=None, stream=None, rule: int = SCALE_FP32,
                   amax_floor: float = 0.0, scale_floor: float = 0.0) -> None:
    """One read of BF16 x [rows x cols]: its 1x128 cast (q, scales, as
    fp8_quant_1x128) and its 128x1 transposed cast (qT, scalesT, as
    fp8_requant_128x1_T from BF16), optional host group offsets."""
    _dual_common("fp8_quant_dual_opts", x, q, scales, qT, scalesT, offsets, stream, rule, amax_floor,
                 scale_floor)


def fp8_quant_dual_stash(x: torch.Tensor, q: torch.Tensor, scales: torch.Tensor, qT: torch.Tensor,
                         scalesT: torch.Tensor, offsets=None, stream=None, rule: int = SCALE_FP32,
                         amax_floor: float = 0.0, scale_floor: float = 0.0) -> None:
    """One read of BF16 x [rows x cols]: its 1x128 cast (q, scales, as
    fp8_quant_1x128) and the 128x1 transposed requant of that E4M3 result
    (qT, scalesT, as fp8_requant_128x1_T from q, scales), optional host
    group offsets."""
    _dual_common("fp8_quant_dual_stash_opts", x, q, scales, qT, scalesT, offsets, stream, rule, amax_floor,
                 scale_floor)


def fp8_quant_dual_stash_opts(x, q, scales, qT, scalesT, opts: Optional["ScaleOpts"], offsets=None,
                              stream=None) -> None:
    """fp8_quant_dual_stash under the scale rule `opts` (None: default)."""
    fp8_quant_dual_stash(x, q, scales, qT, scalesT, offsets=offsets, stream=stream, **_rule_kwargs(opts))


def fp8_quant_dual_sr(x, q, scales, qT, scalesT, seed: int, salt: int = 0, offsets=None, stream=None,
                      rule: int = SCALE_FP32, amax_floor: float = 0.0, scale_floor: float = 0.0) -> None:
    """fp8_quant_dual with stochastic rounding: the 1x128 part under (seed,
    salt), the transposed part under (seed, salt + 1); see fp8bs.h."""
    _dual_common("fp8_quant_dual_sr", x, q, scales, qT, scalesT, offsets, stream, rule, amax_floor, scale_floor,
                 sr=(seed, salt))


def fp8_quant_dual_stash_sr(x, q, scales, qT, scalesT, seed: int, salt: int = 0, offsets=None, stream=None,
                            rule: int = SCALE_FP32, amax_floor: float = 0.0, scale_floor: float = 0.0) -> None:
    """fp8_quant_dual_stash with stochastic rounding: the 1x128 part under
    (seed, salt), the requant of its result under (seed, salt + 1)."""
    _dual_common("fp8_quant_dual_stash_sr", x, q, scales, qT, scalesT, offsets, stream, rule, amax_floor,
                 scale_floor, sr=(seed, salt))


def _require_dev(offsets):
    if not _on_device(offsets):
        raise ValueError("offsets_dev must be a CUDA int32 tensor")


def fp8_requant_128x1_T_dev(src, src_scales, qT, scalesT, offsets_dev, opts: Optional["ScaleOpts"] = None,
                            stream=None) -> None:
    """fp8_requant_128x1_T with group offsets read on the device (outputs
    sized by empty_requant_128x1_T with the same offsets tensor)."""
    _require_dev(offsets_dev)
    fp8_requant_128x1_T(src, src_scales, qT, scalesT, offsets_dev, stream, **_rule_kwargs(opts))


def fp8_quant_dual_dev(x, q, scales, qT, scalesT, offsets_dev, opts: Optional["ScaleOpts"] = None,
                       stream=None) -> None:
    """fp8_quant_dual with group offsets read on the device."""
    _require_dev(offsets_dev)
    fp8_quant_dual(x, q, scales, qT, scalesT, offsets_dev, stream, **_rule_kwargs(opts))


def fp8_quant_dual_stash_dev(x, q, scales, qT, scalesT, offsets_dev, opts: Optional["ScaleOpts"] = None,
                             stream=None) -> None:
    """fp8_quant_dual_stash with group offsets read on the device."""
    _require_dev(offsets_dev)
    fp8_quant_dual_stash(x, q, scales, qT, scalesT, offsets_dev, stream, **_rule_kwargs(opts))


def _dual_common(fn, x, q, scales, qT, scalesT, offsets, stream, rule, amax_floor, scale_floor, sr=None) -> None:
    _need(x, torch.bfloat16, "x")
    for t, n, d in ((q, "q", torch.uint8), (scales, "scales", torch.float32), (qT, "qT", torch.uint8),
                    (scalesT, "scalesT", torch.float32)):
        _need(t, d, n)
    rows, cols = x.shape
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    if q.shape != (rows, cols) or scales.shape != ((cols + 127) // 128, fp8bs_scale_ld(rows)):
        raise ValueError("q / scales shapes do not match empty_quant_1x128")
    mp = _padded(rows, offsets)
    if qT.shape != (cols, mp) or scalesT.shape != (mp // 128, cols):
        raise ValueError("qT / scalesT shapes do not match empty_requant_128x1_T")
    if _on_device(offsets):
        if sr is not None:
            raise ValueError("stochastic rounding takes host offsets")
        dev_fn = {"fp8_quant_dual_opts": "fp8_quant_dual_dev",
                  "fp8_quant_dual_stash_opts": "fp8_quant_dual_stash_dev"}[fn]
        optr, groups = _offsets_dev(offsets)
        _check(dev_fn, getattr(lib(), dev_fn)(
            _ptr(x), rows, cols, optr, groups, _ptr(q), _ptr(scales), _ptr(qT), _ptr(scalesT),
            _opts(rule, amax_floor, scale_floor), _stream(stream)))
        return
    if offsets is not None:
        off = _offsets_host(offsets)
        optr, groups = off.ctypes.data_as(ctypes.c_void_p), off.size - 1
    else:
        off, optr, groups = None, None, 0
    if sr is None:
        _check(fn[:-len("_opts")], getattr(lib(), fn)(
            _ptr(x), rows, cols, optr, groups, _ptr(q), _ptr(scales), _ptr(qT), _ptr(scalesT),
            _opts(rule, amax_floor, scale_floor), _stream(stream)))
    else:
        _check(fn, getattr(lib(), fn)(
            _ptr(x), rows, cols, optr, groups, _ptr(q), _ptr(scales), _ptr(qT), _ptr(scalesT),
            int(sr[0]) & (2 ** 64 - 1), int(sr[1]) & 0xFFFFFFFF, _opts(rule, amax_floor, scale_floor),
            _stream(stream)))


def fp8_quant_1x128_sr(x, q, scales, seed: int, salt: int = 0, stream=None, rule: int = SCALE_FP32,
                       amax_floor: float = 0.0, scale_floor: float = 0.0) -> None:
    """fp8_quant_1x128 with stochastic rounding under (seed, salt); see fp8bs.h."""
    _need(x, torch.bfloat16, "x"); _need(q, torch.uint8, "q"); _need(scales, torch.float32, "scales")
    rows, cols = x.shape
    if q.shape != (rows, cols) or scales.shape != ((cols + 127) // 128, fp8bs_scale_ld(rows)):
        raise ValueError("output shapes do not match empty_quant_1x128")
    _check("fp8_quant_1x128_sr", lib().fp8_quant_1x128_sr(
        _ptr(x), rows, cols, cols, _ptr(q), _ptr(scales), int(seed) & (2 ** 64 - 1), int(salt) & 0xFFFFFFFF,
        _opts(rule, amax_floor, scale_floor), _stream(stream)))


def fp8_quant_128x128_sr(w, q, qT, scales, seed: int, salt: int = 0, stream=None, rule: int = SCALE_FP32,
                         amax_floor: float = 0.0, scale_floor: float = 0.0) -> None:
    """fp8_quant_128x128 with stochastic rounding under (seed, salt); see fp8bs.h."""
    _need(w, torch.bfloat16, "w"); _need(q, torch.uint8, "q"); _need(scales, torch.float32, "scales")
    if qT is not None:
        _need(qT, torch.uint8, "qT")
    batch = w.shape[0] if w.dim() == 3 else 1
    rows, cols = w.shape[-2:]
    nb = ((rows + 127) // 128) * ((cols + 127) // 128)
    if (q.numel() != w.numel() or q.shape[-2:] != (rows, cols) or scales.numel() != batch * nb
            or (qT is not None and (qT.numel() != w.numel() or qT.shape[-2:] != (cols, rows)))):
        raise ValueError("output shapes do not match empty_quant_128x128")
    _check("fp8_quant_128x128_sr", lib().fp8_quant_128x128_sr(
        _ptr(w), batch, rows, cols, cols, _ptr(q), _ptr(qT), _ptr(scales), int(seed) & (2 ** 64 - 1),
        int(salt) & 0xFFFFFFFF, _opts(rule, amax_floor, scale_floor), _stream(stream)))


def fp8bs_mx_scale_bytes(rows: int, cols: int) -> int:
    return int(lib().fp8bs_mx_scale_bytes(int(rows), int(cols)))


def empty_mx_quant(rows: int, cols: int, device="cuda"):
    """(q uint8 [rows x cols], scale atoms uint8 [fp8bs_mx_scale_bytes])."""
    q = torch.empty((rows, cols), dtype=torch.uint8, device=device)
    sc = torch.empty(max(fp8bs_mx_scale_bytes(rows, cols), 0), dtype=torch.uint8, device=device)
    return q, sc


def fp8_mx_quant_1x32(x, q, scale_atoms, stream=None) -> None:
    """MXFP8 1x32 quantization of BF16 x [rows x cols] (cols % 128 == 0)."""
    _need(x, torch.bfloat16, "x"); _need(q, torch.uint8, "q"); _need(scale_atoms, torch.uint8, "scale_atoms")
    rows, cols = x.shape
    if q.shape != (rows, cols) or scale_atoms.numel() < fp8bs_mx_scale_bytes(rows, cols):
        raise ValueError("output shapes do not match empty_mx_quant")
    _check("fp8_mx_quant_1x32", lib().fp8_mx_quant_1x32(_ptr(x), rows, cols, _ptr(q), _ptr(scale_atoms),
                                                        _stream(stream)))


def fp8_mx_gemm(a, a_atoms, b, b_atoms, out, stream=None) -> None:
    """out [M x N] (BF16, or FP32 through fp8_mx_gemm_f32) = A [M x K] . B [N x K]^T,
    both MXFP8 along K."""
    f32 = out.dtype == torch.float32
    for t, n, d in ((a, "a", torch.uint8), (a_atoms, "a_atoms", torch.uint8), (b, "b", torch.uint8),
                    (b_atoms, "b_atoms", torch.uint8), (out, "out", torch.float32 if f32 else torch.bfloat16)):
        _need(t, d, n)
    M, K = a.shape
    N = b.shape[0]
    if b.shape != (N, K) or out.shape != (M, N):
        raise ValueError("shape mismatch")
    name = "fp8_mx_gemm_f32" if f32 else "fp8_mx_gemm"
    _check(name, getattr(lib(), name)(_ptr(a), _ptr(a_atoms), _ptr(b), _ptr(b_atoms), M, N, K,
                                      _ptr(out), _stream(stream)))


def fp8_mx_gemm_wkn(a, a_atoms, b, b_atoms, out, stream=None) -> None:
    """out [M x N] (BF16) = A [M x K] . B with B's codes [K x N] (W as the
    128x128 cast stores it) and B's atoms in the [N x K] layout."""
    for t, n, d in ((a, "a", torch.uint8), (a_atoms, "a_atoms", torch.uint8), (b, "b", torch.uint8),
                    (b_atoms, "b_atoms", torch.uint8), (out, "out", torch.bfloat16)):
        _need(t, d, n)
    M, K = a.shape
    N = b.shape[1]
    if b.shape != (K, N) or out.shape != (M, N):
        raise ValueError("shape mismatch")
    _check("fp8_mx_gemm_wkn", lib().fp8_mx_gemm_wkn(_ptr(a), _ptr(a_atoms), _ptr(b), _ptr(b_atoms), M, N, K,
                                                    _ptr(out), _stream(stream)))


def fp8_mx_gemm_f32(a, a_atoms, b, b_atoms, out, stream=None) -> None:
    """fp8_mx_gemm with an FP32 output tensor (the Wgrad form)."""
    _need(out, torch.float32, "out")
    fp8_mx_gemm(a, a_atoms, b, b_atoms, out, stream)


def empty_mx_quant_T(rows: int, cols: int, device="cuda"):
    """(qT uint8 [cols x Mpad], scale atoms) for fp8_mx_quant_1x32_T of a
    [rows x cols] tensor; Mpad = 128 * ceil(rows / 128)."""
    mp = (rows + 127) // 128 * 128
    return empty_mx_quant(cols, mp, device)


def fp8_mx_quant_1x32_T(x, qT, scale_atoms, stream=None) -> None:
    """Transposed MXFP8 cast of BF16 x [rows x cols]: 32-row blocks, qT [cols x Mpad]."""
    _need(x, torch.bfloat16, "x"); _need(qT, torch.uint8, "qT"); _need(scale_atoms, torch.uint8, "scale_atoms")
    rows, cols = x.shape
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    mp = (rows + 127) // 128 * 128
    if qT.shape != (cols, mp) or scale_atoms.numel() < fp8bs_mx_scale_bytes(cols, mp):
        raise ValueError("output shapes do not match empty_mx_quant_T")
    _check("fp8_mx_quant_1x32_T", lib().fp8_mx_quant_1x32_T(_ptr(x), rows, cols, _ptr(qT), _ptr(scale_atoms),
                                                            _stream(stream)))


def fp8_pack_ue8m0(scales, rows: int, K: int, row_block: int, row_stride: int, kb_stride: int,
                   scale_atoms, stream=None) -> None:
    """Exponent bytes of power-of-two fp32 block scales into the MX scale
    atoms of an operand [rows x K] (each 128-element K-block's byte repeated
    over its four 32-element blocks). The scale of (row r, K-block b) is
    scales.flatten()[(r // row_block) * row_stride + b * kb_stride]; scales
    that are not powers of two record FP8BS_ERR_DEVICE (fp8bs_device_status)."""
    _need(scales, torch.float32, "scales"); _need(scale_atoms, torch.uint8, "scale_atoms")
    rows, K = int(rows), int(K)
    if rows > 0 and K > 0:
        last = ((rows - 1) // int(row_block)) * int(row_stride) + (K // 128 - 1) * int(kb_stride)
        if not scales.is_contiguous() or last >= scales.numel():
            raise ValueError("scales do not hold every (row, K-block) index")
        if scale_atoms.numel() < fp8bs_mx_scale_bytes(rows, K):
            raise ValueError("scale_atoms smaller than fp8bs_mx_scale_bytes(rows, K)")
    _check("fp8_pack_ue8m0", lib().fp8_pack_ue8m0(_ptr(scales), rows, K, int(row_block), int(row_stride),
                                                  int(kb_stride), _ptr(scale_atoms), _stream(stream)))


def empty_mx_atoms(rows: int, K: int, batch: int = 1, device="cuda"):
    """Scale atoms (uint8) of `batch` operands [rows x K] for the MX GEMM."""
    return torch.empty(batch * max(fp8bs_mx_scale_bytes(rows, K), 0), dtype=torch.uint8, device=device)


def fp8_quant_128x128_packed(w, q, qT, scales, atoms_wT, atoms_w, stream=None) -> None:
    """fp8_quant_128x128 under the UE8M0 rule that also writes the scale atoms
    of W^T [cols x rows] (atoms_wT) and of W [rows x cols] (atoms_w), per
    batch entry; rows, cols multiples of 128. qT may be None (no transposed
    codes: the MX Fprop then reads q through fp8_mx_gemm_wkn)."""
    _need(w, torch.bfloat16, "w"); _need(q, torch.uint8, "q"); _need(scales, torch.float32, "scales")
    if qT is not None:
        _need(qT, torch.uint8, "qT")
    _need(atoms_wT, torch.uint8, "atoms_wT"); _need(atoms_w, torch.uint8, "atoms_w")
    batch = w.shape[0] if w.dim() == 3 else 1
    rows, cols = w.shape[-2:]
    nb = ((rows + 127) // 128) * ((cols + 127) // 128)
    if (q.numel() != w.numel() or q.shape[-2:] != (rows, cols) or scales.numel() != batch * nb
            or (qT is not None and (qT.numel() != w.numel() or qT.shape[-2:] != (cols, rows)))):
        raise ValueError("output shapes do not match empty_quant_128x128")
    need = batch * fp8bs_mx_scale_bytes(cols, rows)
    if atoms_wT.numel() < need or atoms_w.numel() < need:
        raise ValueError("atoms smaller than batch * fp8bs_mx_scale_bytes(cols, rows)")
    _check("fp8_quant_128x128_packed", lib().fp8_quant_128x128_packed(
        _ptr(w), batch, rows, cols, cols, _ptr(q), _ptr(qT), _ptr(scales), _ptr(atoms_wT), _ptr(atoms_w),
        _opts(SCALE_UE8M0, 0.0, 0.0), _stream(stream)))


def _dual_packed(fn, x, q, scales, qT, scalesT, q_atoms, qT_atoms, stream, offsets=None) -> None:
    _need(x, torch.bfloat16, "x")
    for t, n, d in ((q, "q", torch.uint8), (scales, "scales", torch.float32), (qT, "qT", torch.uint8),
                    (scalesT, "scalesT", torch.float32), (q_atoms, "q_atoms", torch.uint8),
                    (qT_atoms, "qT_atoms", torch.uint8)):
        _need(t, d, n)
    rows, cols = x.shape
    if not x.is_contiguous():
        raise ValueError("x must be contiguous")
    mp = _padded(rows, offsets)
    if (q.shape != (rows, cols) or scales.shape != ((cols + 127) // 128, fp8bs_scale_ld(rows))
            or qT.shape != (cols, mp) or scalesT.shape != (mp // 128, cols)):
        raise ValueError("output shapes do not match empty_quant_1x128 / empty_requant_128x1_T")
    q_rows = rows if offsets is None else mp      # grouped: the groups' tile layout
    if q_atoms.numel() < fp8bs_mx_scale_bytes(q_rows, cols) or qT_atoms.numel() < fp8bs_mx_scale_bytes(cols, mp):
        raise ValueError("atoms smaller than fp8bs_mx_scale_bytes of q / qT")
    opts = _opts(SCALE_UE8M0, 0.0, 0.0)
    if offsets is None:
        _check(fn, getattr(lib(), fn)(_ptr(x), rows, cols, _ptr(q), _ptr(scales), _ptr(qT), _ptr(scalesT),
                                      _ptr(q_atoms), _ptr(qT_atoms), opts, _stream(stream)))
        return
    dptr, hptr, groups, _, keep = _offsets_args(offsets, rows, rows)
    gfn = fn + "_grouped"
    _check(gfn, getattr(lib(), gfn)(_ptr(x), rows, cols, dptr, hptr, groups, _ptr(q), _ptr(scales), _ptr(qT),
                                    _ptr(scalesT), _ptr(q_atoms), _ptr(qT_atoms), opts, _stream(stream)))
    del keep


def fp8_quant_dual_packed(x, q, scales, qT, scalesT, q_atoms, qT_atoms, stream=None, offsets=None) -> None:
    """fp8_quant_dual under the UE8M0 rule that also writes the scale atoms
    of q [rows x cols] and of qT [cols x Mpad], cols % 128 == 0. With
    ``offsets`` (host sequence or CUDA tensor, as in fp8_quant_dual) the
    grouped form: q's atoms in the groups' tile layout."""
    _dual_packed("fp8_quant_dual_packed", x, q, scales, qT, scalesT, q_atoms, qT_atoms, stream, offsets)


def fp8_quant_dual_stash_packed(x, q, scales, qT, scalesT, q_atoms, qT_atoms, stream=None, offsets=None) -> None:
    """fp8_quant_dual_stash under the UE8M0 rule that also writes the scale
    atoms of q [rows x cols] and of qT [cols x Mpad], cols % 128 == 0. With
    ``offsets``, the grouped form (see fp8_quant_dual_packed)."""
    _dual_packed("fp8_quant_dual_stash_packed", x, q, scales, qT, scalesT, q_atoms, qT_atoms, stream, offsets)


def fp8_quant_dual_packed_grouped(x, q, scales, qT, scalesT, q_atoms, qT_atoms, offsets, stream=None) -> None:
    """The grouped form of fp8_quant_dual_packed (offsets required)."""
    if offsets is None:
        raise ValueError("the grouped form needs offsets")
    fp8_quant_dual_packed(x, q, scales, qT, scalesT, q_atoms, qT_atoms, stream, offsets)


def fp8_quant_dual_stash_packed_grouped(x, q, scales, qT, scalesT, q_atoms, qT_atoms, offsets,
                                        stream=None) -> None:
    """The grouped form of fp8_quant_dual_stash_packed (offsets required)."""
    if offsets is None:
        raise ValueError("the grouped form needs offsets")
    fp8_quant_dual_stash_packed(x, q, scales, qT, scalesT, q_atoms, qT_atoms, stream, offsets)


def _rule_kwargs(opts: Optional[ScaleOpts]) -> dict:
    if opts is None:
        return {}
    return dict(rule=int(opts.rule), amax_floor=float(opts.amax_floor), scale_floor=float(opts.scale_floor))


def fp8_quant_1x128_opts(x, q, scales, opts: Optional[ScaleOpts], stream=None) -> None:
    """fp8_quant_1x128 under the scale rule `opts` (None: default)."""
    fp8_quant_1x128(x, q, scales, stream=stream, **_rule_kwargs(opts))


def fp8_quant_128x128_opts(w, q, qT, scales, opts: Optional[ScaleOpts], stream=None) -> None:
    """fp8_quant_128x128 under the scale rule `opts` (None: default)."""
    fp8_quant_128x128(w, q, qT, scales, stream=stream, **_rule_kwargs(opts))


def fp8_requant_128x1_T_opts(src, src_scales, qT, scalesT, opts: Optional[ScaleOpts], offsets=None,
                             stream=None) -> None:
    """fp8_requant_128x1_T under the scale rule `opts` (None: default)."""
    fp8_requant_128x1_T(src, src_scales, qT, scalesT, offsets=offsets, stream=stream, **_rule_kwargs(opts))


def fp8_quant_dual_opts(x, q, scales, qT, scalesT, opts: Optional[ScaleOpts], offsets=None,
                        stream=None) -> None:
    """fp8_quant_dual under the scale rule `opts` (None: default)."""
    fp8_quant_dual(x, q, scales, qT, scalesT, offsets=offsets, stream=stream, **_rule_kwargs(opts))


def fp8_block_gemm_fprop(xq, sx, wqT, sw, y, stream=None) -> None:
    """Y[M x N] (BF16) = X W from xq [M x K], sx, wqT [N x K], sw [K/128 x N/128]."""
    for t, n, d in ((xq, "xq", torch.uint8), (sx, "sx", torch.float32), (wqT, "wqT", torch.uint8),
                    (sw, "sw", torch.float32), (y, "y", torch.bfloat16)):
        _need(t, d, n)
    M, K = xq.shape
    N = wqT.shape[0]
    if wqT.shape != (N, K) or y.shape != (M, N):
        raise ValueError("shape mismatch")
    _check("fp8_block_gemm_fprop", lib().fp8_block_gemm_fprop(
        _ptr(xq), _ptr(sx), _ptr(wqT), _ptr(sw), M, N, K, _ptr(y), _stream(stream)))


def fp8_block_gemm_fprop_wkn(xq, sx, wq, sw, y, stream=None) -> None:
    """Y[M x N] (BF16) = X W from xq [M x K], sx, wq [K x N] (W's codes as
    the 128x128 cast wrote them), sw [K/128 x N/128]."""
    for t, n, d in ((xq, "xq", torch.uint8), (sx, "sx", torch.float32), (wq, "wq", torch.uint8),
                    (sw, "sw", torch.float32), (y, "y", torch.bfloat16)):
        _need(t, d, n)
    M, K = xq.shape
    N = wq.shape[1]
    if wq.shape != (K, N) or y.shape != (M, N):
        raise ValueError("shape mismatch")
    _check("fp8_block_gemm_fprop_wkn", lib().fp8_block_gemm_fprop_wkn(
        _ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw), M, N, K, _ptr(y), _stream(stream)))


def fp8_block_gemm_dgrad(dyq, sdy, wq, sw, dx, stream=None) -> None:
    """dX[M x K] (BF16) = dY W^T from dyq [M x N], sdy, wq [K x N], sw."""
    for t, n, d in ((dyq, "dyq", torch.uint8), (sdy, "sdy", torch.float32), (wq, "wq", torch.uint8),
                    (sw, "sw", torch.float32), (dx, "dx", torch.bfloat16)):
        _need(t, d, n)
    M, N = dyq.shape
    K = wq.shape[0]
    if wq.shape != (K, N) or dx.shape != (M, K):
        raise ValueError("shape mismatch")
    _check("fp8_block_gemm_dgrad", lib().fp8_block_gemm_dgrad(
        _ptr(dyq), _ptr(sdy), _ptr(wq), _ptr(sw), M, N, K, _ptr(dx), _stream(stream)))


def fp8_block_gemm_wgrad(dyqT, sdyT, xqT, sxT, dw, accumulate: bool = False, stream=None) -> None:
    """dW[N x K] (FP32) = dY^T X from dyqT [N x T], sdyT [T/128 x N], xqT [K x T], sxT [T/128 x K]."""
    for t, n, d in ((dyqT, "dyqT", torch.uint8), (sdyT, "sdyT", torch.float32),
                    (xqT, "xqT", torch.uint8), (sxT, "sxT", torch.float32), (dw, "dw", torch.float32)):
        _need(t, d, n)
    N, T = dyqT.shape
    K = xqT.shape[0]
    if xqT.shape != (K, T) or dw.shape != (N, K):
        raise ValueError("shape mismatch")
    _check("fp8_block_gemm_wgrad", lib().fp8_block_gemm_wgrad(
        _ptr(dyqT), _ptr(sdyT), _ptr(xqT), _ptr(sxT), T, N, K, _ptr(dw), int(bool(accumulate)),
        _stream(stream)))


def fp8_block_gemm_grouped(op: int, offsets, a, sa, b, sb, out, N: int, K: int,
                           accumulate: bool = False, stream=None, rows: Optional[int] = None) -> None:
    """Grouped (MoE) GEMM; see fp8bs.h for the operand layouts of each op.

    ``offsets`` (groups + 1 int32 row offsets) given as a CUDA tensor is read
    by the kernel on the device (nothing is copied to the host, so the call
    can sit in a CUDA graph whose routing changes between replays); any other
    sequence is a host array. ``rows`` is the total token count: by default
    a.shape[0] for Fprop / Dgrad and offsets[-1] for Wgrad with host offsets;
    Wgrad with device offsets needs it."""
    for t, n, d in ((a, "a", torch.uint8), (sa, "sa", torch.float32), (b, "b", torch.uint8),
                    (sb, "sb", torch.float32)):
        _need(t, d, n)
    _need(out, torch.float32 if op == OP_WGRAD else torch.bfloat16, "out")
    if _on_device(offsets):
        dptr, groups = _offsets_dev(offsets)
        hptr = None
        if rows is None:
            if op == OP_WGRAD:
                raise ValueError("Wgrad with device offsets needs rows (the total token count)")
            rows = a.shape[0]
    else:
        off = _offsets_host(offsets)
        dptr, hptr, groups = None, off.ctypes.data_as(ctypes.c_void_p), off.size - 1
        if rows is None:
            rows = int(off[-1])
    _check("fp8_block_gemm_grouped", lib().fp8_block_gemm_grouped(
        int(op), groups, dptr, hptr, int(rows), _ptr(a), _ptr(sa), _ptr(b),
        _ptr(sb), int(N), int(K), _ptr(out), int(bool(accumulate)), _stream(stream)))


def _offsets_args(offsets, rows, default_rows):
    """(device pointer, host pointer, groups, rows, keepalive) of an offsets argument."""
    if _on_device(offsets):
        dptr, groups = _offsets_dev(offsets)
        if rows is None:
            if default_rows is None:
                raise ValueError("device offsets need rows (the total token count)")
            rows = default_rows
        return dptr, None, groups, int(rows), None
    off = _offsets_host(offsets)
    if rows is None:
        rows = int(off[-1])
    return None, off.ctypes.data_as(ctypes.c_void_p), off.size - 1, int(rows), off


def fp8_mx_gemm_grouped(op: int, offsets, a, a_atoms, b, b_atoms, out, N: int, K: int, stream=None,
                        rows: Optional[int] = None) -> None:
    """Grouped (MoE) MX GEMM; see fp8bs.h for the operand and atom layouts of
    each op. Offsets as in fp8_block_gemm_grouped (a CUDA tensor is read on
    the device); rows defaults to a.shape[0] for Fprop / Dgrad."""
    for t, n in ((a, "a"), (a_atoms, "a_atoms"), (b, "b"), (b_atoms, "b_atoms")):
        _need(t, torch.uint8, n)
    _need(out, torch.float32 if op == OP_WGRAD else torch.bfloat16, "out")
    dptr, hptr, groups, rows, keep = _offsets_args(offsets, rows, None if op == OP_WGRAD else a.shape[0])
    _check("fp8_mx_gemm_grouped", lib().fp8_mx_gemm_grouped(
        int(op), groups, dptr, hptr, rows, _ptr(a), _ptr(a_atoms), _ptr(b), _ptr(b_atoms), int(N), int(K),
        _ptr(out), _stream(stream)))
    del keep


def fp8_pack_ue8m0_grouped(scales, rows: int, K: int, offsets, atoms, stream=None) -> None:
    """Exponent bytes of the 1x128 power-of-two scales [K/128 x scale_ld] of
    grouped rows [rows x K] into the groups' tile layout of the MX atoms."""
    _need(scales, torch.float32, "scales")
    _need(atoms, torch.uint8, "atoms")
    dptr, hptr, groups, rows, keep = _offsets_args(offsets, rows, rows)
    _check("fp8_pack_ue8m0_grouped", lib().fp8_pack_ue8m0_grouped(
        _ptr(scales), rows, int(K), int(scales.shape[1]), groups, dptr, hptr, _ptr(atoms), _stream(stream)))
    del keep


def _splitk_dims(op: int, a, b):
    """(M, N, K) of a split-K call from its operands (see fp8bs.h)."""
    if op == OP_FPROP:      # a = xq [M x K], b = wqT [N x K]
        M, K = a.shape
        N = b.shape[0]
        if b.shape != (N, K):
            raise ValueError("shape mismatch")
        return M, N, K, (M, N)
    if op == OP_FPROP_WKN:  # a = xq [M x K], b = wq [K x N]
        M, K = a.shape
        N = b.shape[1]
        if b.shape != (K, N):
            raise ValueError("shape mismatch")
        return M, N, K, (M, N)
    if op == OP_DGRAD:      # a = dyq [M x N], b = wq [K x N]
        M, N = a.shape
        K = b.shape[0]
        if b.shape != (K, N):
            raise ValueError("shape mismatch")
        return M, N, K, (M, K)
    raise ValueError("split-K supports OP_FPROP, OP_FPROP_WKN and OP_DGRAD")


def fp8bs_splitk_workspace_size(op: int, M: int, N: int, K: int, splits: int) -> int:
    return int(lib().fp8bs_splitk_workspace_size(int(op), int(M), int(N), int(K), int(splits)))


def fp8bs_splitk_default_splits(op: int, M: int, N: int, K: int) -> int:
    return int(lib().fp8bs_splitk_default_splits(int(op), int(M), int(N), int(K)))


def fp8_block_gemm_splitk(op: int, a, sa, b, sb, out, splits: Optional[int] = None,
                          workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    """Split-K Fprop (a = xq, b = wqT; OP_FPROP_WKN: b = wq) or Dgrad (a = dyq,
    b = wq) into BF16 `out`.

    `splits` defaults to fp8bs_splitk_default_splits. `workspace` is a device
    buffer of at least fp8bs_splitk_workspace_size bytes; if None, one is
    allocated here with torch (memory plumbing only)."""
    for t, n, d in ((a, "a", torch.uint8), (sa, "sa", torch.float32), (b, "b", torch.uint8),
                    (sb, "sb", torch.float32), (out, "out", torch.bfloat16)):
        _need(t, d, n)
    M, N, K, out_shape = _splitk_dims(op, a, b)
    if tuple(out.shape) != out_shape:
        raise ValueError("shape mismatch")
    if splits is None:
        splits = fp8bs_splitk_default_splits(op, M, N, K)
    need = fp8bs_splitk_workspace_size(op, M, N, K, splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=a.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("fp8_block_gemm_splitk", lib().fp8_block_gemm_splitk(
        int(op), _ptr(a), _ptr(sa), _ptr(b), _ptr(sb), M, N, K, int(splits), _ptr(out),
        _ptr(workspace), wbytes, _stream(stream)))


def fp8_block_gemm_splitk_noalloc(op: int, a, sa, b, sb, out, splits: Optional[int] = None,
                                  stream=None) -> None:
    """fp8_block_gemm_splitk with the library's fixed scratch array instead of
    a workspace (for callers that cannot allocate; see fp8bs.h for the size
    limit and the rule that overlapping calls must be serialized)."""
    for t, n, d in ((a, "a", torch.uint8), (sa, "sa", torch.float32), (b, "b", torch.uint8),
                    (sb, "sb", torch.float32), (out, "out", torch.bfloat16)):
        _need(t, d, n)
    M, N, K, out_shape = _splitk_dims(op, a, b)
    if tuple(out.shape) != out_shape:
        raise ValueError("shape mismatch")
    if splits is None:
        splits = fp8bs_splitk_default_splits(op, M, N, K)
    need = fp8bs_splitk_workspace_size(op, M, N, K, splits)
    detail = ""
    if need > NOALLOC_SCRATCH_BYTES:
        detail = (f"{splits} ranges of {M} x {out_shape[1]} fp32 need {need} bytes, more than the fixed "
                  f"{NOALLOC_SCRATCH_BYTES}-byte scratch; use fewer splits or fp8_block_gemm_splitk "
                  "with a workspace")
    _check("fp8_block_gemm_splitk_noalloc", lib().fp8_block_gemm_splitk_noalloc(
        int(op), _ptr(a), _ptr(sa), _ptr(b), _ptr(sb), M, N, K, int(splits), _ptr(out),
        _stream(stream)), detail)


def fp8bs_device_status(reset: bool = True) -> int:
    """Synchronize and return the device status word (0 = OK)."""
    return int(lib().fp8bs_device_status(int(bool(reset))))


def fp8bs_last_device_status(stream=None, reset: bool = False) -> int:
    """The device status word as of the work issued so far on `stream`
    (waits for that stream only, not the whole device)."""
    return int(lib().fp8bs_last_device_status(_stream(stream), int(bool(reset))))


def fp8bs_copy_device_status(dst: torch.Tensor, reset: bool = False, stream=None) -> None:
    """Enqueue a copy of the device status word into dst (a CUDA int32 tensor
    of one element) on `stream`, without waiting; capturable in a graph."""
    _need(dst, torch.int32, "dst")
    if dst.numel() != 1:
        raise ValueError("dst: one int32 element")
    _check("fp8bs_copy_device_status", lib().fp8bs_copy_device_status(_ptr(dst), int(bool(reset)),
                                                                       _stream(stream)))


def fp8bs_set_wait_limit_ns(ns: int) -> None:
    lib().fp8bs_set_wait_limit_ns(int(ns))


def fp8bs_selftest_wait_timeout(limit_ns: int, stream=None) -> None:
    _check("fp8bs_selftest_wait_timeout",
           lib().fp8bs_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def fp8bs_selftest_gemm_timeout(xq, sx, wqT, sw, y, limit_ns: int, stream=None) -> None:
    """fp8_block_gemm_fprop with the epilogue holding its buffers and every
    wait bounded by limit_ns: records FP8BS_ERR_TIMEOUT (test hook)."""
    for t, n, d in ((xq, "xq", torch.uint8), (sx, "sx", torch.float32), (wqT, "wqT", torch.uint8),
                    (sw, "sw", torch.float32), (y, "y", torch.bfloat16)):
        _need(t, d, n)
    M, K = xq.shape
    N = wqT.shape[0]
    if wqT.shape != (N, K) or y.shape != (M, N):
        raise ValueError("shape mismatch")
    _check("fp8bs_selftest_gemm_timeout", lib().fp8bs_selftest_gemm_timeout(
        _ptr(xq), _ptr(sx), _ptr(wqT), _ptr(sw), M, N, K, _ptr(y), int(limit_ns), _stream(stream)))
