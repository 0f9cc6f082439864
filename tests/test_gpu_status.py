"""Failure detection on the GPU without a fault: a bounded wait on a barrier
that nothing arrives on gives up, records FP8BS_ERR_TIMEOUT in the device
status word, and the context stays usable for the next kernels."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs
import oracle
import workloads as wl
from parity import np_, u16

pytestmark = pytest.mark.gpu

ERR_TIMEOUT = 5


def test_bounded_wait_reports_timeout_and_context_survives():
    fp8bs.build()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    fp8bs.fp8bs_selftest_wait_timeout(2_000_000)      # 2 ms
    assert fp8bs.fp8bs_device_status(reset=False) == ERR_TIMEOUT
    assert fp8bs.fp8bs_device_status(reset=True) == ERR_TIMEOUT
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    # the context is still usable
    x = wl.normal((64, 256), seed=1)
    q, s = fp8bs.empty_quant_1x128(64, 256)
    fp8bs.fp8_quant_1x128(x.cuda(), q, s)
    torch.cuda.synchronize()
    oq, _ = oracle.quant_1x128(u16(x))
    assert np.array_equal(np_(q), oq)
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def test_invalid_arguments_raise_before_launch():
    fp8bs.build()
    x = torch.zeros((4, 24), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((4, 24), dtype=torch.uint8, device="cuda")
    s = torch.empty((1, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(fp8bs.Fp8bsError) as e:
        fp8bs.fp8_quant_1x128(x, q, s)
    assert e.value.code == 3



def _fprop_case(M, K, N, seed):
    x = wl.normal((M, K), seed=seed)
    w = wl.normal((K, N), std=wl.W_STD, seed=seed + 1)
    xq, sx = fp8bs.empty_quant_1x128(M, K)
    fp8bs.fp8_quant_1x128(x.cuda(), xq, sx)
    wq, wqT, sw = fp8bs.empty_quant_128x128(K, N)
    fp8bs.fp8_quant_128x128(w.cuda(), wq, wqT, sw)
    return xq, sx, wq, wqT, sw


def test_gemm_wait_timeout_aborts_cleanly_and_the_next_gemm_is_exact():
    """A real GEMM whose bounded wait gives up: the self-test form of Fprop
    keeps the epilogue from handing tensor-memory buffers back, so the MMA
    thread's wait for the third K-block's buffer runs out after the limit.
    The kernel records FP8BS_ERR_TIMEOUT, stops issuing, drains its copies
    and MMAs, frees its tensor memory and returns; the context stays usable
    and the same GEMM, launched normally, matches the oracle."""
    fp8bs.build()
    M, K, N = 256, 1024, 512
    xq, sx, wq, wqT, sw = _fprop_case(M, K, N, seed=11)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8bs_selftest_gemm_timeout(xq, sx, wqT, sw, y, 2_000_000)     # 2 ms
    assert fp8bs.fp8bs_device_status(reset=False) == ERR_TIMEOUT
    assert fp8bs.fp8bs_device_status(reset=True) == ERR_TIMEOUT
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    # twice in a row: the aborted launch left nothing behind (tensor memory
    # freed, barriers private to the launch)
    fp8bs.fp8bs_selftest_gemm_timeout(xq, sx, wqT, sw, y, 2_000_000)
    assert fp8bs.fp8bs_device_status(reset=True) == ERR_TIMEOUT
    # the context is still usable and the next launch is correct
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_fprop(xq, sx, wqT, sw, y)
    torch.cuda.synchronize()
    assert fp8bs.fp8bs_device_status(reset=True) == 0
    from parity import assert_gemm_close, bf16_values, dequant_blocks, dequant_rows
    a = np.abs(dequant_rows(np_(xq), np_(sx)))
    b = np.abs(dequant_blocks(np_(wq), np_(sw)))
    want = oracle.fprop(np_(xq), np_(sx), np_(wq), np_(sw))
    assert_gemm_close(bf16_values(y), want, a @ b, True, "fprop after an aborted launch")
