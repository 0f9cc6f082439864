"""fp8_block_gemm_splitk_noalloc, called through the C ABI: the split-K GEMM
whose range sums live in the library's fixed scratch array, for callers that
cannot allocate device memory (an allocator-free runtime, a loop that must
not call cudaMalloc because it may synchronize the device, a plugin without
a memory pool).

Two calls in a row on the same operands are each byte-identical to
fp8_block_gemm_splitk with a caller workspace and the same split count, and
within the GEMM tolerance |d| <= 2e-3 * sum_k |a_k b_k| + 1e-6 (plus one BF16
ulp) of the oracle's promoted GEMM. Around a call after the first, neither
torch's allocator nor the device's free memory changes. A request larger
than the scratch is rejected with FP8BS_ERR_SHAPE before any work. The file
sorts last so the test also runs after every other GPU test in the same
process; it passes alone in a fresh process as well."""
import ctypes

import numpy as np
import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs
import oracle
import workloads as wl
from parity import assert_gemm_close, bf16_values, dequant_blocks, dequant_rows, np_

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fp8bs.build()
    fp8bs.lib()
    torch.cuda.init()
    yield
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def _quantize(x, w):
    xq, sx = fp8bs.empty_quant_1x128(*x.shape)
    fp8bs.fp8_quant_1x128(x.cuda(), xq, sx)
    wq, wqT, sw = fp8bs.empty_quant_128x128(*w.shape)
    fp8bs.fp8_quant_128x128(w.cuda(), wq, wqT, sw)
    return xq, sx, wq, wqT, sw


def _check_two_calls(op, a, sa, b, sb, out_shape, splits, want, absprod, what):
    ref = torch.empty(out_shape, dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_splitk(op, a, sa, b, sb, ref, splits=splits)
    torch.cuda.synchronize()
    ref_bits = np_(ref.view(torch.int16))
    assert_gemm_close(bf16_values(ref), want, absprod, True, f"{what}, workspace call")
    for call in range(2):
        y = torch.full(out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()
        alloc0 = torch.cuda.memory_allocated()
        free0, _ = torch.cuda.mem_get_info()
        fp8bs.fp8_block_gemm_splitk_noalloc(op, a, sa, b, sb, y, splits=splits)
        torch.cuda.synchronize()
        if call > 0:   # the first call on a device may load the module and look up the scratch
            assert torch.cuda.memory_allocated() == alloc0, what
            assert torch.cuda.mem_get_info()[0] == free0, what
        assert np.array_equal(np_(y.view(torch.int16)), ref_bits), f"{what}, call {call + 1}"
        assert_gemm_close(bf16_values(y), want, absprod, True, f"{what}, call {call + 1}")


def test_noalloc_fprop_long_k_matches_workspace_call_and_oracle():
    d = wl.longk(16384)
    xq, sx, wq, wqT, sw = _quantize(d["X"], d["W"])
    splits = fp8bs.fp8bs_splitk_default_splits(fp8bs.OP_FPROP, 256, 256, 16384)
    assert splits > 1
    assert fp8bs.fp8bs_splitk_workspace_size(fp8bs.OP_FPROP, 256, 256, 16384, splits) <= fp8bs.NOALLOC_SCRATCH_BYTES
    a = np.abs(dequant_rows(np_(xq), np_(sx)))
    b = np.abs(dequant_blocks(np_(wq), np_(sw)))
    want = oracle.fprop(np_(xq), np_(sx), np_(wq), np_(sw))
    _check_two_calls(fp8bs.OP_FPROP, xq, sx, wqT, sw, (256, 256), splits, want, a @ b,
                     "noalloc fprop 256x16384x256")


def test_noalloc_dgrad_matches_workspace_call_and_oracle():
    dy = wl.with_outliers((300, 2048), fraction=0.01, seed=5)
    w = wl.normal((384, 2048), std=wl.W_STD, seed=6)
    dyq, sdy, wq, _, sw = _quantize(dy, w)
    a = np.abs(dequant_rows(np_(dyq), np_(sdy)))
    b = np.abs(dequant_blocks(np_(wq), np_(sw)))
    want = oracle.dgrad(np_(dyq), np_(sdy), np_(wq), np_(sw))
    _check_two_calls(fp8bs.OP_DGRAD, dyq, sdy, wq, sw, (300, 384), 8, want, a @ b.T,
                     "noalloc dgrad 300x2048x384")


def test_noalloc_rejects_requests_larger_than_the_scratch():
    # 8 ranges of a 4096 x 2048 fp32 output need 256 MiB
    M, N, K, splits = 4096, 2048, 7168, 8
    assert fp8bs.fp8bs_splitk_workspace_size(fp8bs.OP_FPROP, M, N, K, splits) > fp8bs.NOALLOC_SCRATCH_BYTES
    null = ctypes.c_void_p(0)
    rc = fp8bs.lib().fp8_block_gemm_splitk_noalloc(fp8bs.OP_FPROP, null, null, null, null, M, N, K, splits,
                                                   null, null)
    assert rc == 3   # FP8BS_ERR_SHAPE
    xq, sx = fp8bs.empty_quant_1x128(M, K)
    wq, wqT, sw = fp8bs.empty_quant_128x128(K, N)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8bs.Fp8bsError, match="fixed") as e:
        fp8bs.fp8_block_gemm_splitk_noalloc(fp8bs.OP_FPROP, xq, sx, wqT, sw, y, splits=splits)
    assert e.value.code == 3
