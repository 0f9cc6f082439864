"""The benchmarked steps captured in CUDA graphs (the form bench.py times):
every entry point they call is capture-safe, and replaying the graph gives
byte-identical outputs to launching the same kernels one by one on one
stream. The dense step's graph runs its two independent pairs (the W and X
casts, Dgrad and Wgrad) on two streams; the long-contraction workload's
graph runs its four problems side by side on their own streams."""
import os
import sys

import pytest
import torch

import fp8_block_scaled_act_gb300 as fp8bs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fp8bs.build()
    fp8bs.lib()
    torch.cuda.init()
    yield
    assert fp8bs.fp8bs_device_status(reset=True) == 0


def _outputs(step):
    # (the step's weight cast writes no transposed codes: Fprop reads W as stored)
    return (step.Y, step.dX, step.dW, step.xq, step.sx, step.xT, step.sxT, step.wq, step.sw,
            step.dyq, step.sdy, step.dyT, step.sdyT)


@pytest.mark.parametrize("M,K,N", [(512, 1024, 512), (384, 768, 256)])
def test_graph_replay_matches_stream_launches(M, K, N):
    dev = torch.device("cuda", 0)
    step = bench.DenseStep(fp8bs, torch, dev, M, K, N, seed=3)
    for f in step.launches():
        f()
    torch.cuda.synchronize()
    ref = [t.clone() for t in _outputs(step)]
    for t in _outputs(step):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run_dag()
    torch.cuda.synchronize()
    for t in _outputs(step):          # capture runs nothing: the outputs are still zero
        t.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, _outputs(step)):
        assert torch.equal(a, b)


def test_longk_graph_with_concurrent_problems_matches_stream_launches():
    dev = torch.device("cuda", 0)
    step = bench.LongKStep(fp8bs, torch, dev, seed=5)
    outs = lambda: [t for c in step.cases for t in (c["Y"], c["xq"], c["sx"], c["wq"], c["sw"])]
    for f in step.launches():
        f()
    torch.cuda.synchronize()
    ref = [t.clone() for t in outs()]
    for t in outs():
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step.run_dag()
    torch.cuda.synchronize()
    for t in outs():
        t.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref, outs()):
        assert torch.equal(a, b)
