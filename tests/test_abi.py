"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports
every function declared in include/fp8bs.h, and its host-side logic (shape
helpers, argument validation that runs before any device work) behaves as
documented. No kernel is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

import fp8_block_scaled_act_gb300 as fp8bs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


@pytest.fixture(scope="module")
def L():
    fp8bs.build()
    return fp8bs.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([A-Za-z_0-9]+)\s*\(", text)
    skip = {"if", "sizeof", "defined"}
    return sorted({n for n in names if n.startswith("fp8") and n not in skip})


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ["fp8_quant_1x128", "fp8_quant_128x128", "fp8_requant_128x1_T",
              "fp8_block_gemm_fprop", "fp8_block_gemm_dgrad", "fp8_block_gemm_wgrad",
              "fp8_block_gemm_grouped", "fp8bs_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in _declared_functions():
        assert hasattr(L, n), n
        assert n in fp8bs.__all__, n


def test_host_helpers(L):
    assert fp8bs.fp8bs_version() >= 100
    assert fp8bs.fp8bs_status_str(0) == "ok"
    assert fp8bs.fp8bs_status_str(5) == "device wait timed out"
    assert [fp8bs.fp8bs_scale_ld(r) for r in (0, 1, 4, 5, 4096)] == [0, 4, 4, 8, 4096]
    assert fp8bs.fp8bs_padded_tokens(0) == 0
    assert fp8bs.fp8bs_padded_tokens(1) == 128
    assert fp8bs.fp8bs_padded_tokens(4096) == 4096
    assert fp8bs.fp8bs_padded_tokens(400, [0, 0, 129, 130, 130, 400]) == 256 + 128 + 384
    with pytest.raises(ValueError):
        fp8bs.fp8bs_padded_tokens(10, [0, 5, 3, 10])       # decreasing
    with pytest.raises(ValueError):
        fp8bs.fp8bs_padded_tokens(10, [0, 5, 9])           # does not end at rows


def test_padded_tokens_max_bounds_every_split():
    """The capacity of the device-offset layouts: 128 floor((rows + 127 k) / 128)
    with k = min(groups, rows) is at least the padded count of every split of
    rows into groups, and reached by some split."""
    g = np.random.default_rng(1)
    assert fp8bs.fp8bs_padded_tokens_max(0, 32) == 0
    assert fp8bs.fp8bs_padded_tokens_max(1, 32) == 128
    assert fp8bs.fp8bs_padded_tokens_max(300, 1) == 384
    assert fp8bs.fp8bs_padded_tokens_max(8192, 32) == 128 * ((8192 + 127 * 32) // 128)
    with pytest.raises(ValueError):
        fp8bs.fp8bs_padded_tokens_max(-1, 2)
    for _ in range(200):
        G = int(g.integers(1, 40))
        rows = int(g.integers(0, 2000))
        cap = fp8bs.fp8bs_padded_tokens_max(rows, G)
        cuts = np.sort(g.integers(0, rows + 1, size=G - 1))
        off = np.concatenate([[0], cuts, [rows]]).astype(np.int32)
        assert fp8bs.fp8bs_padded_tokens(rows, off) <= cap
    # reached: k - 1 groups of 1 token, the rest in the last group
    for rows, G in ((1000, 8), (129, 4), (5, 9)):
        k = min(G, rows)
        counts = [1] * (k - 1) + [rows - (k - 1)] + [0] * (G - k)
        off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        assert fp8bs.fp8bs_padded_tokens(rows, off) == fp8bs.fp8bs_padded_tokens_max(rows, G)


def test_padded_tokens_agrees_with_oracle_geometry():
    import oracle
    g = np.random.default_rng(0)
    for _ in range(20):
        counts = g.integers(0, 300, size=g.integers(1, 40))
        off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        assert fp8bs.fp8bs_padded_tokens(int(off[-1]), off) == oracle.padded_tokens(int(off[-1]), off)


def test_argument_validation_before_device_work(L):
    """Invalid shapes and pointers are rejected on the host, before any CUDA call."""
    P = ctypes.c_void_p
    buf = ctypes.create_string_buffer(1 << 12)
    a16 = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    mis = ctypes.c_void_p(a16.value + 4)
    ERR_ARG, ERR_ALIGN, ERR_SHAPE = 1, 2, 3
    # quant 1x128
    assert L.fp8_quant_1x128(a16, 4, 24, 24, a16, a16, None) == ERR_SHAPE   # cols % 16
    assert L.fp8_quant_1x128(a16, -1, 32, 32, a16, a16, None) == ERR_ARG
    assert L.fp8_quant_1x128(a16, 4, 32, 16, a16, a16, None) == ERR_ARG     # ld < cols
    assert L.fp8_quant_1x128(None, 4, 32, 32, a16, a16, None) == ERR_ARG
    assert L.fp8_quant_1x128(mis, 4, 32, 32, a16, a16, None) == ERR_ALIGN
    assert L.fp8_quant_1x128(a16, 0, 32, 32, None, None, None) == 0         # empty: no work
    # quant 128x128
    assert L.fp8_quant_128x128(a16, 1, 24, 32, 32, a16, None, a16, None) == ERR_SHAPE
    assert L.fp8_quant_128x128(a16, 0, 32, 32, 32, a16, None, a16, None) == ERR_ARG
    assert L.fp8_quant_128x128(a16, 1, 32, 32, 32, a16, mis, a16, None) == ERR_ALIGN
    # requant
    assert L.fp8_requant_128x1_T(7, a16, None, 4, 32, None, 0, a16, a16, None) == ERR_ARG
    assert L.fp8_requant_128x1_T(1, a16, None, 4, 32, None, 0, a16, a16, None) == ERR_ARG  # Q needs scales
    bad = (ctypes.c_int32 * 3)(0, 5, 3)
    assert L.fp8_requant_128x1_T(0, a16, None, 3, 32, bad, 2, a16, a16, None) == ERR_ARG
    # gemms
    assert L.fp8_block_gemm_fprop(a16, a16, a16, a16, 128, 256, 100, a16, None) == ERR_SHAPE
    assert L.fp8_block_gemm_fprop(a16, a16, a16, a16, 128, 200, 128, a16, None) == ERR_SHAPE
    assert L.fp8_block_gemm_fprop(a16, a16, a16, a16, 0, 256, 128, None, None) == 0
    assert L.fp8_block_gemm_fprop(mis, a16, a16, a16, 8, 256, 128, a16, None) == ERR_ALIGN
    assert L.fp8_block_gemm_dgrad(a16, a16, a16, a16, 8, 100, 128, a16, None) == ERR_SHAPE
    assert L.fp8_block_gemm_wgrad(a16, a16, a16, a16, 100, 128, 128, a16, 0, None) == ERR_SHAPE
    assert L.fp8_block_gemm_wgrad(a16, a16, a16, a16, 128, 128, 128, None, 0, None) == ERR_ARG
    off = (ctypes.c_int32 * 3)(0, 4, 8)
    # fp8_block_gemm_grouped(op, groups, offsets_dev, offsets_host, rows, a, sa, b, sb, N, K, out, acc, stream)
    G = L.fp8_block_gemm_grouped
    assert G(9, 2, None, off, 8, a16, a16, a16, a16, 128, 128, a16, 0, None) == ERR_ARG
    assert G(0, 0, None, off, 8, a16, a16, a16, a16, 128, 128, a16, 0, None) == ERR_ARG
    assert G(0, 300, None, off, 8, a16, a16, a16, a16, 128, 128, a16, 0, None) == ERR_ARG
    assert G(0, 2, None, off, 8, a16, a16, a16, a16, 128, 100, a16, 0, None) == ERR_SHAPE
    assert G(0, 2, None, off, 9, a16, a16, a16, a16, 128, 128, a16, 0, None) == ERR_ARG   # rows != off[2]
    assert G(0, 2, a16, off, 8, a16, a16, a16, a16, 128, 128, a16, 0, None) == ERR_ARG    # both offsets
    assert G(0, 2, None, None, 8, a16, a16, a16, a16, 128, 128, a16, 0, None) == ERR_ARG  # neither
    assert G(0, 2, ctypes.c_void_p(a16.value + 2), None, 8, a16, a16, a16, a16, 128, 128, a16, 0,
             None) == ERR_ALIGN
    assert G(0, 2, a16, None, -1, a16, a16, a16, a16, 128, 128, a16, 0, None) == ERR_ARG
    # casts with device offsets: offsets required, no host offsets, groups in range
    R = L.fp8_requant_128x1_T_dev
    assert R(0, a16, None, 8, 32, None, 2, a16, a16, None, None) == ERR_ARG
    assert R(0, a16, None, 8, 32, a16, 0, a16, a16, None, None) == ERR_ARG
    assert R(0, a16, None, 8, 32, a16, 300, a16, a16, None, None) == ERR_ARG
    assert R(0, a16, None, 8, 32, ctypes.c_void_p(a16.value + 2), 2, a16, a16, None, None) == ERR_ALIGN
    for f in (L.fp8_quant_dual_dev, L.fp8_quant_dual_stash_dev):
        assert f(a16, 8, 32, None, 2, a16, a16, a16, a16, None, None) == ERR_ARG
        assert f(a16, 8, 32, a16, 2, None, a16, a16, a16, None, None) == ERR_ARG
        assert f(a16, 8, 24, a16, 2, a16, a16, a16, a16, None, None) == ERR_SHAPE


def test_product_path_does_not_import_oracle():
    """The CUDA path's Python package never references the oracle."""
    pkg = os.path.join(ROOT, "fp8_block_scaled_act_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "fp8bs_oracle" not in text, f


def test_splitk_workspace_arithmetic_and_argument_errors():
    """Workspace size = ranges actually used x one 128 x 256 fp32 slot per
    output tile (ceil(M / 128) x ceil(width / 256) tiles) x 4 bytes, with
    ranges = ceil(nblocks / ceil(nblocks / splits)); bad arguments are
    rejected before any device work."""
    L = fp8bs.lib()
    ws = fp8bs.fp8bs_splitk_workspace_size
    assert ws(fp8bs.OP_FPROP, 256, 256, 65536, 76) == 74 * 256 * 256 * 4    # 512 blocks: 7 per range
    assert ws(fp8bs.OP_FPROP, 256, 256, 1024, 1) == 0
    assert ws(fp8bs.OP_FPROP, 256, 256, 1024, 100) == 8 * 256 * 256 * 4     # clamped to 8 blocks
    assert ws(fp8bs.OP_DGRAD, 256, 256, 1024, 4) == 2 * 256 * 1024 * 4      # contraction N = 256
    assert ws(fp8bs.OP_FPROP, 300, 384, 1024, 4) == 4 * (3 * 2) * 128 * 256 * 4   # ragged: whole tiles
    assert ws(fp8bs.OP_WGRAD, 256, 256, 1024, 4) == 0
    assert ws(fp8bs.OP_FPROP, 0, 256, 1024, 4) == 0
    assert ws(fp8bs.OP_FPROP, 100, 256, 1000, 4) == 0                        # K % 128 != 0
    null = ctypes.c_void_p(0)
    assert L.fp8_block_gemm_splitk(7, null, null, null, null, 128, 128, 128, 2, null, null, 0, null) == 1
    assert L.fp8_block_gemm_splitk(0, null, null, null, null, 128, 128, 128, 0, null, null, 0, null) == 1
    assert L.fp8_block_gemm_splitk(0, null, null, null, null, 128, 100, 128, 2, null, null, 0, null) == 3


def test_ue8m0_packing_argument_validation(L):
    """The packing entries reject bad arguments on the host: the packing's row
    block, shapes, pointers and alignment; the packed casts' rule (UE8M0
    only), shapes and atom pointers."""
    buf = ctypes.create_string_buffer(1 << 12)
    a16 = ctypes.c_void_p((ctypes.addressof(buf) + 15) & ~15)
    mis16 = ctypes.c_void_p(a16.value + 4)
    mis4 = ctypes.c_void_p(a16.value + 2)
    ERR_ARG, ERR_ALIGN, ERR_SHAPE = 1, 2, 3
    # fp8_pack_ue8m0(scales, rows, K, row_block, row_stride, kb_stride, atoms, stream)
    assert L.fp8_pack_ue8m0(a16, 128, 256, 64, 1, 4, a16, None) == ERR_ARG      # row block 1 or 128
    assert L.fp8_pack_ue8m0(a16, 128, 200, 1, 1, 4, a16, None) == ERR_SHAPE    # K % 128
    assert L.fp8_pack_ue8m0(a16, -1, 256, 1, 1, 4, a16, None) == ERR_ARG
    assert L.fp8_pack_ue8m0(a16, 128, 256, 1, -1, 4, a16, None) == ERR_ARG
    assert L.fp8_pack_ue8m0(None, 128, 256, 1, 1, 4, a16, None) == ERR_ARG
    assert L.fp8_pack_ue8m0(a16, 128, 256, 1, 1, 4, mis16, None) == ERR_ALIGN
    assert L.fp8_pack_ue8m0(mis4, 128, 256, 1, 1, 4, a16, None) == ERR_ALIGN
    assert L.fp8_pack_ue8m0(a16, 0, 256, 1, 1, 4, None, None) == 0             # empty: no work
    ue = ctypes.pointer(fp8bs.ScaleOpts(fp8bs.SCALE_UE8M0, 0.0, 0.0))
    f32 = ctypes.pointer(fp8bs.ScaleOpts(fp8bs.SCALE_FP32, 0.0, 0.0))
    # fp8_quant_128x128_packed(w, batch, rows, cols, ldw, q, qT, scales, atoms_wT, atoms_w, opts, stream)
    q2 = L.fp8_quant_128x128_packed
    assert q2(a16, 1, 128, 128, 128, a16, a16, a16, a16, a16, None, None) == ERR_ARG   # rule required
    assert q2(a16, 1, 128, 128, 128, a16, a16, a16, a16, a16, f32, None) == ERR_ARG
    assert q2(a16, 1, 96, 128, 128, a16, a16, a16, a16, a16, ue, None) == ERR_SHAPE     # rows % 128
    assert q2(a16, 1, 128, 128, 128, a16, a16, a16, None, a16, ue, None) == ERR_ARG
    assert q2(a16, 1, 128, 128, 128, a16, a16, a16, a16, mis16, ue, None) == ERR_ALIGN
    # fp8_quant_dual_packed / _stash_packed(x, rows, cols, q, s, qT, sT, q_atoms, qT_atoms, opts, stream)
    for f in (L.fp8_quant_dual_packed, L.fp8_quant_dual_stash_packed):
        assert f(a16, 4, 128, a16, a16, a16, a16, a16, a16, None, None) == ERR_ARG
        assert f(a16, 4, 96, a16, a16, a16, a16, a16, a16, ue, None) == ERR_SHAPE      # cols % 128
        assert f(a16, 4, 128, a16, a16, a16, a16, None, a16, ue, None) == ERR_ARG
        assert f(a16, 4, 128, a16, a16, a16, a16, a16, mis16, ue, None) == ERR_ALIGN
    # the grouped forms (x, rows, cols, offsets_dev, offsets_host, groups, q, s, qT, sT, q_atoms, qT_atoms,
    # opts, stream): exactly one offsets array, the UE8M0 rule, cols % 128
    off = (ctypes.c_int32 * 3)(0, 2, 4)
    for f in (L.fp8_quant_dual_packed_grouped, L.fp8_quant_dual_stash_packed_grouped):
        assert f(a16, 4, 128, None, None, 2, a16, a16, a16, a16, a16, a16, ue, None) == ERR_ARG
        assert f(a16, 4, 128, a16, off, 2, a16, a16, a16, a16, a16, a16, ue, None) == ERR_ARG
        assert f(a16, 4, 128, None, off, 2, a16, a16, a16, a16, a16, a16, f32, None) == ERR_ARG
        assert f(a16, 4, 96, None, off, 2, a16, a16, a16, a16, a16, a16, ue, None) == ERR_SHAPE
        assert f(a16, 4, 128, None, off, 2, a16, a16, a16, a16, None, a16, ue, None) == ERR_ARG
