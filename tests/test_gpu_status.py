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
