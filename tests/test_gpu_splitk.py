"""GPU parity of split-K Fprop / Dgrad (fp8_block_gemm_splitk) against the
CPU oracle, within the GEMM tolerance
    |gpu - oracle| <= 2e-3 * sum_k |a_k b_k| + 1e-6  (+ one BF16 ulp),
on the same GPU-quantized operands as the unsplit tests (checked bit-exact
against the oracle's quantization). Also: one range reproduces the unsplit
kernel bit for bit, results do not depend on scheduling, and a short
workspace is rejected."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs
import oracle
import workloads as wl
from parity import assert_gemm_close, bf16_values, dequant_blocks, dequant_rows, sample_indices
from test_gpu_gemm import q128, q128_oracle, q1x128

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fp8bs.build()
    fp8bs.lib()
    torch.cuda.init()
    yield
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def _fprop_operands(M, K, N, seed):
    x = wl.with_outliers((M, K), fraction=0.01, seed=seed)
    w = wl.normal((K, N), std=wl.W_STD, seed=seed + 1)
    xq, sx, oxq, osx = q1x128(x)
    wq, wqT, sw = q128(w)
    owq, osw = q128_oracle(w)
    return (xq, sx, wqT, sw), (oxq, osx, owq, osw)


def _splitk(op, a, sa, b, sb, out_shape, splits, workspace=None):
    out = torch.empty(out_shape, dtype=torch.bfloat16, device="cuda")
    fp8bs.fp8_block_gemm_splitk(op, a, sa, b, sb, out, splits=splits, workspace=workspace)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("M,K,N,splits", [(300, 1024, 256, 2), (300, 1024, 256, 3), (129, 2048, 384, 7),
                                          (1, 896, 128, 5), (256, 1024, 256, 8), (64, 512, 512, 40)])
def test_splitk_fprop_small(M, K, N, splits):
    (xq, sx, wqT, sw), (oxq, osx, owq, osw) = _fprop_operands(M, K, N, seed=M + K + splits)
    y = bf16_values(_splitk(fp8bs.OP_FPROP, xq, sx, wqT, sw, (M, N), splits))
    ref = oracle.fprop(oxq, osx, owq, osw)
    a, b = dequant_rows(oxq, osx), dequant_blocks(owq, osw)
    assert_gemm_close(y, ref, np.abs(a) @ np.abs(b), True, f"split-K fprop {M}x{K}x{N} / {splits}")


@pytest.mark.parametrize("M,N,K,splits", [(200, 1024, 384, 2), (129, 2048, 256, 16)])
def test_splitk_dgrad_small(M, N, K, splits):
    dy = wl.with_outliers((M, N), fraction=0.01, seed=M + N)
    w = wl.normal((K, N), std=wl.W_STD, seed=K)
    dyq, sdy, odyq, osdy = q1x128(dy)
    wq, _, sw = q128(w)
    owq, osw = q128_oracle(w)
    dx = bf16_values(_splitk(fp8bs.OP_DGRAD, dyq, sdy, wq, sw, (M, K), splits))
    ref = oracle.dgrad(odyq, osdy, owq, osw)
    a, b = dequant_rows(odyq, osdy), dequant_blocks(owq, osw)
    assert_gemm_close(dx, ref, np.abs(a) @ np.abs(b).T, True, f"split-K dgrad {M}x{N}x{K} / {splits}")


def test_splitk_one_range_is_the_unsplit_kernel():
    (xq, sx, wqT, sw), _ = _fprop_operands(300, 1024, 256, seed=7)
    y1 = _splitk(fp8bs.OP_FPROP, xq, sx, wqT, sw, (300, 256), 1)
    y0 = torch.empty_like(y1)
    fp8bs.fp8_block_gemm_fprop(xq, sx, wqT, sw, y0)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


def test_splitk_is_deterministic():
    (xq, sx, wqT, sw), _ = _fprop_operands(256, 4096, 256, seed=11)
    a = _splitk(fp8bs.OP_FPROP, xq, sx, wqT, sw, (256, 256), 13)
    b = _splitk(fp8bs.OP_FPROP, xq, sx, wqT, sw, (256, 256), 13)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_splitk_rejects_short_workspace():
    (xq, sx, wqT, sw), _ = _fprop_operands(128, 1024, 128, seed=3)
    need = fp8bs.fp8bs_splitk_workspace_size(fp8bs.OP_FPROP, 128, 128, 1024, 4)
    assert need == 4 * 128 * 256 * 4     # one 128 x 256 tile slot per range
    short = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8bs.Fp8bsError):
        _splitk(fp8bs.OP_FPROP, xq, sx, wqT, sw, (128, 128), 4, workspace=short)


def test_splitk_default_splits_fill_the_gpu():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # two 128x256 output tiles and 512 K-blocks: one range per SM
    assert fp8bs.fp8bs_splitk_default_splits(fp8bs.OP_FPROP, 256, 256, 65536) == sms // 2
    # 32 K-blocks: at least four per range; 8 K-blocks: not worth a split
    assert fp8bs.fp8bs_splitk_default_splits(fp8bs.OP_FPROP, 256, 256, 4096) == 8
    assert fp8bs.fp8bs_splitk_default_splits(fp8bs.OP_FPROP, 256, 256, 1024) == 1
    assert fp8bs.fp8bs_splitk_default_splits(fp8bs.OP_FPROP, 4096, 2048, 7168) == 1


@pytest.mark.parametrize("K", wl.LONGK_VALUES)
def test_splitk_longk_default(K):
    """The long-K drift workload (256 x K x 256, U(0.5, 1.5)) with the default
    split: sampled outputs plus a full tile against the oracle."""
    d = wl.longk(K)
    xq, sx, oxq, osx = q1x128(d["X"])
    wq, wqT, sw = q128(d["W"])
    owq, osw = q128_oracle(d["W"])
    splits = fp8bs.fp8bs_splitk_default_splits(fp8bs.OP_FPROP, 256, 256, K)
    y = bf16_values(_splitk(fp8bs.OP_FPROP, xq, sx, wqT, sw, (256, 256), splits))
    ii, jj = sample_indices(256, 256, 512, seed=K, tiles=((0, 0),))
    ref = oracle.fprop(oxq, osx, owq, osw, ii, jj)
    truth, _ = oracle.fprop_reference_sums(oxq, osx, owq, osw, ii, jj, unpromoted=False)
    assert_gemm_close(y[ii, jj], ref, np.abs(truth), True, f"split-K longk {K} / {splits}")
