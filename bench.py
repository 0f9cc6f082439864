"""Benchmark of the fine-grained FP8 linear layer on GB300.

One step is one pass of the layer's whole data path over one batch of
synthetic input: the weight's 128x128 quantization (codes and scales; Fprop
reads the codes as stored), the 1x128 quantization of X, Fprop, the
dual-orientation cast of dY
(its 1x128 and 128x1 transposed quantizations from one read), Dgrad, the
128x1 transposed requant of X from its E4M3 stash, and Wgrad. Default workload: X 4096x7168 (N(0,1) with 0.1% outliers),
W 7168x2048 (N(0,0.02^2)), dY 4096x2048 (N(0,1e-3^2)); its numbers are the
line's headline keys. After it the default run times, each the same way and
reported under its own key of ``configs``: the same dense step with
power-of-two scales on the block-scaled MMA, the grouped MoE expert pass (32
experts, 8192 routed rows, group offsets in device memory) with fp32 and
with power-of-two scales, the 256 x K x 256 split-K Fprop of the
long-contraction workload (K = 1024 ... 65536) and the standalone 1x128 cast
of a 16384 x 16384 tensor (``--dense-only`` skips them).
``--workload moe|moe_ue8m0|longk|quant16k|dense_ue8m0`` times one of those as
the headline instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timing: W untimed warm-up steps, then exactly K steps, each one replay of a
CUDA graph of the step (--no-graph: stream launches) bracketed by CUDA
events on the launching stream, with an L2 flush (a 256 MiB write) between
steps outside the events; a second pass of K steps launched kernel by kernel
with an event after every kernel gives the per-kernel table and the
roofline figures. Under torchrun each rank runs its own replica (weak
scaling, no collective on the data path); the step time is the max over
ranks. Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 block-scaled GEMM TFLOP/s (% FP8 peak); quantize GB/s (% HBM BW)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 2.0    # nominal dense ratio (4.5 / 2.25 PFLOP/s)
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------------------
# workload description (shared by both arms)
# ---------------------------------------------------------------------------

def dense_shapes():
    return {"M": 4096, "K": 7168, "N": 2048}


def step_work(M, K, N):
    """Algorithmic FLOPs of the three GEMMs and algorithmic bytes of each
    kernel of one dense step (bytes read + written, scales included)."""
    gemm_flops = 2.0 * M * N * K
    s_ld = (M + 3) // 4 * 4
    b = {
        "quant_128x128(W)": K * N * 2 + K * N + 4 * (K // 128) * (N // 128),
        "quant_dual_stash(X)": M * K * 2 + M * K + 4 * (K // 128) * s_ld + M * K + 4 * (M // 128) * K,
        "fprop": M * K + N * K + 4 * (K // 128) * (s_ld + N // 128) + 2 * M * N,
        "quant_dual(dY)": M * N * 2 + M * N + 4 * (N // 128) * s_ld + M * N + 4 * (M // 128) * N,
        "dgrad": M * N + K * N + 4 * (N // 128) * s_ld + 4 * (K // 128) * (N // 128) + 2 * M * K,
        "wgrad": N * M + K * M + 4 * (M // 128) * (N + K) + 4 * N * K,
    }
    flops = {"fprop": gemm_flops, "dgrad": gemm_flops, "wgrad": gemm_flops}
    return flops, b


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# distributed plumbing (host logic; gloo-testable on CPU)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device="cpu") -> float:
    """Max of a per-rank float over all ranks (identity without a group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(per_rank_work: float, world: int, max_seconds: float) -> float:
    """Work all ranks processed divided by the slowest rank's time."""
    return per_rank_work * world / max_seconds


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

def smi_gpu_id(local: int) -> str:
    """nvidia-smi's id for this rank's GPU (CUDA_VISIBLE_DEVICES remaps indices)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [v for v in sm if mx and v >= 0.3 * max(mx)]
        return {"sm_mhz": statistics.median(loaded or sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class DenseStep:
    """Buffers and the launch sequence of one dense fwd+bwd step."""

    def __init__(self, fp8bs, torch, device, M, K, N, seed=0):
        self.fp8bs, self.torch, self.dev = fp8bs, torch, device
        self.M, self.K, self.N = M, K, N
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        X = torch.randn(M, K, device=device, generator=g)
        n_out = int(round(1e-3 * M * K))
        pos = torch.randperm(M * K, device=device, generator=g)[:n_out]
        mag = torch.rand(n_out, device=device, generator=g) * 150.0 + 50.0
        sgn = torch.where(torch.rand(n_out, device=device, generator=g) < 0.5, -1.0, 1.0)
        X.view(-1)[pos] = mag * sgn
        self.X = X.to(torch.bfloat16)
        self.W = (torch.randn(K, N, device=device, generator=g) * 0.02).to(torch.bfloat16)
        self.dY = (torch.randn(M, N, device=device, generator=g) * 1e-3).to(torch.bfloat16)
        e = fp8bs
        self.xq, self.sx = e.empty_quant_1x128(M, K, device)
        # Fprop reads W's codes as stored ([K x N], MN-major), so the cast
        # writes no transposed copy
        self.wq, self.wqT, self.sw = e.empty_quant_128x128(K, N, with_transpose=False, device=device)
        self.Y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
        self.dyq, self.sdy = e.empty_quant_1x128(M, N, device)
        self.dX = torch.empty(M, K, dtype=torch.bfloat16, device=device)
        self.xT, self.sxT = e.empty_requant_128x1_T(M, K, device=device)
        self.dyT, self.sdyT = e.empty_requant_128x1_T(M, N, device=device)
        self.dW = torch.empty(N, K, dtype=torch.float32, device=device)
        self.names = ["quant_128x128(W)", "quant_dual_stash(X)", "fprop", "quant_dual(dY)", "dgrad", "wgrad"]
        self.side = torch.cuda.Stream(device)
        self.dag_desc = "CUDA graph, two streams (W || X casts, Dgrad || Wgrad)"

    def work(self):
        return step_work(self.M, self.K, self.N)

    def io(self):
        return (self.X, self.W, self.dY), (self.Y, self.dX, self.dW)

    def describe(self):
        M, K, N = self.M, self.K, self.N
        return {"workload": f"dense FP8 linear fwd+bwd X {M}x{K}, W {K}x{N}, dY {M}x{N}",
                "M": M, "K": K, "N": N}

    def launches(self):
        e = self.fp8bs
        return [
            lambda: e.fp8_quant_128x128(self.W, self.wq, None, self.sw),
            # the forward cast of X also writes the Wgrad operand: the 128x1
            # transposed requant of its E4M3 stash
            lambda: e.fp8_quant_dual_stash(self.X, self.xq, self.sx, self.xT, self.sxT),
            lambda: e.fp8_block_gemm_fprop_wkn(self.xq, self.sx, self.wq, self.sw, self.Y),
            lambda: e.fp8_quant_dual(self.dY, self.dyq, self.sdy, self.dyT, self.sdyT),
            lambda: e.fp8_block_gemm_dgrad(self.dyq, self.sdy, self.wq, self.sw, self.dX),
            lambda: e.fp8_block_gemm_wgrad(self.dyT, self.sdyT, self.xT, self.sxT, self.dW),
        ]


    def run_dag(self):
        """The step with its two independent pairs on two streams: the W and
        X casts of the forward, then Dgrad and Wgrad of the backward."""
        torch, L = self.torch, self.launches_cached()
        main = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        self.side.wait_event(fork)
        with torch.cuda.stream(self.side):
            L[0]()                                  # W cast
        w_done = torch.cuda.Event()
        w_done.record(self.side)
        L[1]()                                      # X cast + stash requant
        main.wait_event(w_done)
        L[2]()                                      # Fprop
        L[3]()                                      # dY dual cast
        dy_done = torch.cuda.Event()
        dy_done.record(main)
        self.side.wait_event(dy_done)
        with torch.cuda.stream(self.side):
            L[5]()                                  # Wgrad
        wg_done = torch.cuda.Event()
        wg_done.record(self.side)
        L[4]()                                      # Dgrad
        main.wait_event(wg_done)

    def launches_cached(self):
        if not hasattr(self, "_launches"):
            self._launches = self.launches()
        return self._launches


class DenseUe8m0Step(DenseStep):
    """The dense step with power-of-two scales: the same casts under the
    UE8M0 scale rule, each also writing its scales as exponent bytes in the
    layout the MX GEMM reads (the *_packed casts), and the three GEMMs run on
    the tensor core's block scaling (the MX kernel) instead of the software
    promotion."""

    def __init__(self, fp8bs, torch, device, M, K, N, seed=0):
        super().__init__(fp8bs, torch, device, M, K, N, seed)
        e = fp8bs
        Mp = self.xT.shape[1]
        atoms = lambda rows, k: torch.empty(e.fp8bs_mx_scale_bytes(rows, k), dtype=torch.uint8, device=device)
        self.ax, self.awT, self.ady = atoms(M, K), atoms(N, K), atoms(M, N)
        self.aw, self.adyT, self.axT = atoms(K, N), atoms(N, Mp), atoms(K, Mp)
        self.names = ["quant_128x128(W)+atoms", "quant_dual_stash(X)+atoms", "mx_fprop", "quant_dual(dY)+atoms",
                      "mx_dgrad", "mx_wgrad"]

    def work(self):
        M, K, N = self.M, self.K, self.N
        flops, b = step_work(M, K, N)
        Mp = self.xT.shape[1]
        atoms = lambda rows, k: rows * k // 32                            # exponent bytes of an operand
        bytes_ = {
            "quant_128x128(W)+atoms": b["quant_128x128(W)"] + atoms(N, K) + atoms(K, N),
            "quant_dual_stash(X)+atoms": b["quant_dual_stash(X)"] + atoms(M, K) + atoms(K, Mp),
            "mx_fprop": M * K + N * K + atoms(M, K) + atoms(N, K) + 2 * M * N,
            "quant_dual(dY)+atoms": b["quant_dual(dY)"] + atoms(M, N) + atoms(N, Mp),
            "mx_dgrad": M * N + K * N + atoms(M, N) + atoms(K, N) + 2 * M * K,
            "mx_wgrad": N * Mp + K * Mp + atoms(N, Mp) + atoms(K, Mp) + 4 * N * K,
        }
        f = flops["fprop"]
        return {"mx_fprop": f, "mx_dgrad": f, "mx_wgrad": f}, bytes_

    def describe(self):
        d = super().describe()
        d["workload"] = (d["workload"] + ", power-of-two (UE8M0) scales, GEMMs on the tensor core's block "
                         "scaling over exponent bytes the casts write")
        return d

    def launches(self):
        e = self.fp8bs
        # each cast writes its scales' exponent bytes into the atoms of the
        # GEMM operands it feeds, in the same pass
        return [
            lambda: e.fp8_quant_128x128_packed(self.W, self.wq, None, self.sw, self.awT, self.aw),
            lambda: e.fp8_quant_dual_stash_packed(self.X, self.xq, self.sx, self.xT, self.sxT, self.ax, self.axT),
            lambda: e.fp8_mx_gemm_wkn(self.xq, self.ax, self.wq, self.awT, self.Y),
            lambda: e.fp8_quant_dual_packed(self.dY, self.dyq, self.sdy, self.dyT, self.sdyT, self.ady,
                                            self.adyT),
            lambda: e.fp8_mx_gemm(self.dyq, self.ady, self.wq, self.aw, self.dX),
            lambda: e.fp8_mx_gemm_f32(self.dyT, self.adyT, self.xT, self.axT, self.dW),
        ]


class MoeStep:
    """Grouped MoE expert pass: 1x128 quantization of X, A and dY, batched
    128x128 quantization of the expert weights, Fprop of the up and down
    projections, Dgrad and Wgrad of the down projection (with the grouped
    128x1 requants of dY and A)."""

    def __init__(self, fp8bs, torch, device, tokens=8192, experts=32, hidden=7168, inter=2048,
                 up=4096, seed=0):
        import workloads as wl
        self.fp8bs, self.torch, self.dev = fp8bs, torch, device
        counts = wl.expert_counts(tokens, experts, seed=seed)
        self.offsets_host = wl.offsets_from_counts(counts)
        # the routing lives on the device: the grouped calls read it there, so
        # the captured step needs no host copy of it
        self.offsets = torch.tensor(self.offsets_host, dtype=torch.int32, device=device)
        self.counts = counts
        self.T, self.G, self.H, self.I, self.U = tokens, experts, hidden, inter, up
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        bf = torch.bfloat16
        self.X = torch.randn(tokens, hidden, device=device, generator=g).to(bf)
        self.A = torch.randn(tokens, inter, device=device, generator=g).to(bf)
        self.dY = (torch.randn(tokens, hidden, device=device, generator=g) * 1e-3).to(bf)
        self.Wu = (torch.randn(experts, hidden, up, device=device, generator=g) * 0.02).to(bf)
        self.Wd = (torch.randn(experts, inter, hidden, device=device, generator=g) * 0.02).to(bf)
        e = fp8bs
        self.xq, self.sx = e.empty_quant_1x128(tokens, hidden, device)
        self.aq, self.sa = e.empty_quant_1x128(tokens, inter, device)
        self.dyq, self.sdy = e.empty_quant_1x128(tokens, hidden, device)
        # the grouped Fprops read the experts' codes as stored (MN-major), so
        # the batched casts write no transposed copies
        self.wuq, self.wuqT, self.swu = e.empty_quant_128x128(hidden, up, batch=experts, with_transpose=False,
                                                              device=device)
        self.wdq, self.wdqT, self.swd = e.empty_quant_128x128(inter, hidden, batch=experts, with_transpose=False,
                                                              device=device)
        self.Yu = torch.empty(tokens, up, dtype=bf, device=device)
        self.Yd = torch.empty(tokens, hidden, dtype=bf, device=device)
        self.dA = torch.empty(tokens, inter, dtype=bf, device=device)
        self.dyT, self.sdyT = e.empty_requant_128x1_T(tokens, hidden, self.offsets, device)
        self.aT, self.saT = e.empty_requant_128x1_T(tokens, inter, self.offsets, device)
        self.dWd = torch.empty(experts, hidden, inter, dtype=torch.float32, device=device)
        self.names = ["quant_128x128(W_up)", "quant_128x128(W_down)", "quant_1x128(X)",
                      "grouped_fprop_up", "quant_dual_stash(A)", "grouped_fprop_down", "quant_dual(dY)",
                      "grouped_dgrad_down", "grouped_wgrad_down"]

    def work(self):
        T, G, H, I, U = self.T, self.G, self.H, self.I, self.U
        s_ld = (T + 3) // 4 * 4
        mp = int(self.fp8bs.fp8bs_padded_tokens(T, self.offsets_host))
        flops = {"grouped_fprop_up": 2.0 * T * H * U, "grouped_fprop_down": 2.0 * T * I * H,
                 "grouped_dgrad_down": 2.0 * T * H * I, "grouped_wgrad_down": 2.0 * T * H * I}
        b = {
            "quant_128x128(W_up)": G * H * U * 3 + 4 * G * (H // 128) * (U // 128),
            "quant_128x128(W_down)": G * I * H * 3 + 4 * G * (I // 128) * (H // 128),
            "quant_1x128(X)": T * H * 3 + 4 * (H // 128) * s_ld,
            "grouped_fprop_up": T * H + G * U * H + 2 * T * U,
            "quant_dual_stash(A)": T * I * 3 + 4 * (I // 128) * s_ld + I * mp + 4 * (mp // 128) * I,
            "grouped_fprop_down": T * I + G * H * I + 2 * T * H,
            "quant_dual(dY)": T * H * 3 + 4 * (H // 128) * s_ld + H * mp + 4 * (mp // 128) * H,
            "grouped_dgrad_down": T * H + G * I * H + 2 * T * I,
            "grouped_wgrad_down": (H + I) * mp + 4 * G * H * I,
        }
        return flops, b

    def launches(self):
        e, off, G, H, I, U = self.fp8bs, self.offsets, self.G, self.H, self.I, self.U
        return [
            lambda: e.fp8_quant_128x128(self.Wu, self.wuq, None, self.swu),
            lambda: e.fp8_quant_128x128(self.Wd, self.wdq, None, self.swd),
            lambda: e.fp8_quant_1x128(self.X, self.xq, self.sx),
            lambda: e.fp8_block_gemm_grouped(e.OP_FPROP_WKN, off, self.xq, self.sx, self.wuq, self.swu,
                                             self.Yu, U, H),
            lambda: e.fp8_quant_dual_stash(self.A, self.aq, self.sa, self.aT, self.saT, offsets=off),
            lambda: e.fp8_block_gemm_grouped(e.OP_FPROP_WKN, off, self.aq, self.sa, self.wdq, self.swd,
                                             self.Yd, H, I),
            lambda: e.fp8_quant_dual(self.dY, self.dyq, self.sdy, self.dyT, self.sdyT, offsets=off),
            lambda: e.fp8_block_gemm_grouped(e.OP_DGRAD, off, self.dyq, self.sdy, self.wdq, self.swd,
                                             self.dA, H, I),
            lambda: e.fp8_block_gemm_grouped(e.OP_WGRAD, off, self.dyT, self.sdyT, self.aT, self.saT,
                                             self.dWd, H, I, rows=self.T),
        ]

    def io(self):
        return (self.X, self.A, self.dY, self.Wu, self.Wd), (self.Yu, self.Yd, self.dA, self.dWd)

    def describe(self):
        return {"workload": (f"grouped MoE experts: {self.G} experts, {self.T} routed rows "
                             f"(Dirichlet(0.5) counts), W_up {self.H}x{self.U}, W_down {self.I}x{self.H}; "
                             "group offsets in device memory"),
                "experts": self.G, "tokens": self.T, "hidden": self.H, "inter": self.I, "up": self.U}


class MoeUe8m0Step(MoeStep):
    """The grouped MoE expert pass with power-of-two (UE8M0) scales: the same
    casts under the UE8M0 rule, each writing its scales' exponent bytes into
    the MX scale atoms in the same pass (the weight casts; the grouped dual
    casts of A and dY, in the groups' tile layout; X's 1x128 cast is packed
    by a separate launch), and the four grouped GEMMs on the tensor core's
    block scaling (fp8_mx_gemm_grouped) instead of the software promotion."""

    def __init__(self, fp8bs, torch, device, **kw):
        super().__init__(fp8bs, torch, device, **kw)
        e = fp8bs
        T, G, H, I, U = self.T, self.G, self.H, self.I, self.U
        self.opts = e.ScaleOpts(e.SCALE_UE8M0, 0.0, 0.0)
        cap = int(e.fp8bs_padded_tokens_max(T, G))
        atoms = lambda rows, k, b=1: e.empty_mx_atoms(rows, k, batch=b, device=device)
        self.awuT, self.awu = atoms(U, H, G), atoms(H, U, G)
        self.awdT, self.awd = atoms(H, I, G), atoms(I, H, G)
        self.ax, self.aa, self.ady = atoms(cap, H), atoms(cap, I), atoms(cap, H)
        self.adyT, self.aaT = atoms(H, cap), atoms(I, cap)
        self.cap = cap
        self.names = ["quant_128x128(W_up)+atoms", "quant_128x128(W_down)+atoms", "quant_1x128(X)",
                      "pack(X)", "mx_grouped_fprop_up", "quant_dual_stash(A)+atoms", "mx_grouped_fprop_down",
                      "quant_dual(dY)+atoms", "mx_grouped_dgrad_down", "mx_grouped_wgrad_down"]

    def work(self):
        flops, b = super().work()
        T, G, H, I, U = self.T, self.G, self.H, self.I, self.U
        mp = int(self.fp8bs.fp8bs_padded_tokens(T, self.offsets_host))
        s_ld = (T + 3) // 4 * 4
        f = {"mx_grouped_fprop_up": flops["grouped_fprop_up"], "mx_grouped_fprop_down": flops["grouped_fprop_down"],
             "mx_grouped_dgrad_down": flops["grouped_dgrad_down"], "mx_grouped_wgrad_down": flops["grouped_wgrad_down"]}
        atom = lambda rows, k: rows * k // 32
        by = {
            "quant_128x128(W_up)+atoms": b["quant_128x128(W_up)"] + G * (atom(U, H) + atom(H, U)),
            "quant_128x128(W_down)+atoms": b["quant_128x128(W_down)"] + G * (atom(H, I) + atom(I, H)),
            "quant_1x128(X)": b["quant_1x128(X)"],
            "pack(X)": 4 * (H // 128) * s_ld + atom(mp, H),
            "mx_grouped_fprop_up": b["grouped_fprop_up"] + atom(mp, H) + G * atom(U, H),
            "quant_dual_stash(A)+atoms": b["quant_dual_stash(A)"] + atom(mp, I) + atom(I, mp),
            "mx_grouped_fprop_down": b["grouped_fprop_down"] + atom(mp, I) + G * atom(H, I),
            "quant_dual(dY)+atoms": b["quant_dual(dY)"] + atom(mp, H) + atom(H, mp),
            "mx_grouped_dgrad_down": b["grouped_dgrad_down"] + atom(mp, H) + G * atom(I, H),
            "mx_grouped_wgrad_down": b["grouped_wgrad_down"] + atom(H, mp) + atom(I, mp),
        }
        return f, by

    def launches(self):
        e, off, G, H, I, U, T, o = self.fp8bs, self.offsets, self.G, self.H, self.I, self.U, self.T, self.opts
        return [
            lambda: e.fp8_quant_128x128_packed(self.Wu, self.wuq, None, self.swu, self.awuT, self.awu),
            lambda: e.fp8_quant_128x128_packed(self.Wd, self.wdq, None, self.swd, self.awdT, self.awd),
            lambda: e.fp8_quant_1x128_opts(self.X, self.xq, self.sx, o),
            lambda: e.fp8_pack_ue8m0_grouped(self.sx, T, H, off, self.ax),
            lambda: e.fp8_mx_gemm_grouped(e.OP_FPROP_WKN, off, self.xq, self.ax, self.wuq, self.awuT, self.Yu, U, H),
            lambda: e.fp8_quant_dual_stash_packed(self.A, self.aq, self.sa, self.aT, self.saT, self.aa, self.aaT,
                                                  offsets=off),
            lambda: e.fp8_mx_gemm_grouped(e.OP_FPROP_WKN, off, self.aq, self.aa, self.wdq, self.awdT, self.Yd, H, I),
            lambda: e.fp8_quant_dual_packed(self.dY, self.dyq, self.sdy, self.dyT, self.sdyT, self.ady, self.adyT,
                                            offsets=off),
            lambda: e.fp8_mx_gemm_grouped(e.OP_DGRAD, off, self.dyq, self.ady, self.wdq, self.awd, self.dA, H, I),
            lambda: e.fp8_mx_gemm_grouped(e.OP_WGRAD, off, self.dyT, self.adyT, self.aT, self.aaT, self.dWd, H, I,
                                          rows=T),
        ]

    def describe(self):
        d = super().describe()
        d["workload"] = (d["workload"] + ", power-of-two (UE8M0) scales, the grouped GEMMs on the tensor core's "
                         "block scaling (fp8_mx_gemm_grouped)")
        return d


class LongKStep:
    """The long-contraction drift workload: X 256xK and W Kx256, U(0.5, 1.5),
    for K in 1024, 4096, 16384, 65536; per K the 1x128 and 128x128
    quantizations and a split-K Fprop with the library's default split (two
    128x256 output tiles would otherwise occupy two SMs)."""

    KS = (1024, 4096, 16384, 65536)

    def __init__(self, fp8bs, torch, device, M=256, N=256, seed=0):
        self.fp8bs, self.torch, self.dev = fp8bs, torch, device
        self.M, self.N = M, N
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        e = fp8bs
        self.cases = []
        for K in self.KS:
            X = (torch.rand(M, K, device=device, generator=g) + 0.5).to(torch.bfloat16)
            W = (torch.rand(K, N, device=device, generator=g) + 0.5).to(torch.bfloat16)
            xq, sx = e.empty_quant_1x128(M, K, device)
            wq, wqT, sw = e.empty_quant_128x128(K, N, with_transpose=False, device=device)
            sp = e.fp8bs_splitk_default_splits(e.OP_FPROP_WKN, M, N, K)
            ws = torch.empty(max(16, e.fp8bs_splitk_workspace_size(e.OP_FPROP_WKN, M, N, K, sp)),
                             dtype=torch.uint8, device=device)
            Y = torch.empty(M, N, dtype=torch.bfloat16, device=device)
            self.cases.append(dict(K=K, X=X, W=W, xq=xq, sx=sx, wq=wq, wqT=wqT, sw=sw, sp=sp, ws=ws, Y=Y))
        # the four problems are independent: two streams each (X || W cast)
        self.streams = [torch.cuda.Stream(device) for _ in range(2 * len(self.cases))]
        self.dag_desc = "CUDA graph, the four problems on their own streams (X || W casts, then split-K Fprop)"
        self.names = []
        for c in self.cases:
            self.names += [f"quant_1x128(X,K={c['K']})", f"quant_128x128(W,K={c['K']})",
                           f"splitk_fprop(K={c['K']},splits={c['sp']})"]

    def work(self):
        M, N = self.M, self.N
        s_ld = (M + 3) // 4 * 4
        flops, b = {}, {}
        for c in self.cases:
            K = c["K"]
            b[f"quant_1x128(X,K={K})"] = M * K * 3 + 4 * (K // 128) * s_ld
            b[f"quant_128x128(W,K={K})"] = K * N * 3 + 4 * (K // 128) * (N // 128)
            flops[f"splitk_fprop(K={K},splits={c['sp']})"] = 2.0 * M * N * K
        return flops, b

    def launches(self):
        e = self.fp8bs
        out = []
        for c in self.cases:
            out += [lambda c=c: e.fp8_quant_1x128(c["X"], c["xq"], c["sx"]),
                    lambda c=c: e.fp8_quant_128x128(c["W"], c["wq"], None, c["sw"]),
                    lambda c=c: e.fp8_block_gemm_splitk(e.OP_FPROP_WKN, c["xq"], c["sx"], c["wq"], c["sw"],
                                                        c["Y"], splits=c["sp"], workspace=c["ws"])]
        return out

    def run_dag(self):
        """The problems run side by side, the longest first: each on its own
        stream, its W cast on a second one, so the small problems use SMs the
        large ones leave idle (the split-K GEMMs take one SM per range)."""
        torch, L = self.torch, self.launches_cached()
        main = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(main)
        done = []
        for i in reversed(range(len(self.cases))):
            sx, sw = self.streams[2 * i], self.streams[2 * i + 1]
            sx.wait_event(fork)
            sw.wait_event(fork)
            with torch.cuda.stream(sw):
                L[3 * i + 1]()                      # W cast
            w_done = torch.cuda.Event()
            w_done.record(sw)
            with torch.cuda.stream(sx):
                L[3 * i]()                          # X cast
                sx.wait_event(w_done)
                L[3 * i + 2]()                      # split-K Fprop (and its reduction)
            ev = torch.cuda.Event()
            ev.record(sx)
            done.append(ev)
        for ev in done:
            main.wait_event(ev)

    def launches_cached(self):
        if not hasattr(self, "_launches"):
            self._launches = self.launches()
        return self._launches

    def io(self):
        return (tuple(t for c in self.cases for t in (c["X"], c["W"])),
                tuple(c["Y"] for c in self.cases))

    def describe(self):
        return {"workload": (f"long-K drift workload: X {self.M}xK, W Kx{self.N}, U(0.5,1.5), "
                             f"K in {list(self.KS)}, split-K Fprop"),
                "M": self.M, "N": self.N, "K": list(self.KS)}


class Quant1x128Step:
    """The standalone 1x128 cast of the long-K workload's bandwidth case: a
    16384 x 16384 BF16 N(0, 1) tensor to E4M3 with fp32 scales."""

    def __init__(self, fp8bs, torch, device, R=16384, C=16384, seed=0):
        self.fp8bs, self.torch, self.dev = fp8bs, torch, device
        self.R, self.C = R, C
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.X = torch.randn(R, C, device=device, generator=g).to(torch.bfloat16)
        self.q, self.s = fp8bs.empty_quant_1x128(R, C, device)
        self.names = [f"quant_1x128({R}x{C})"]

    def work(self):
        s_ld = (self.R + 3) // 4 * 4
        return {}, {self.names[0]: self.R * self.C * 3 + 4 * (self.C // 128) * s_ld}

    def launches(self):
        return [lambda: self.fp8bs.fp8_quant_1x128(self.X, self.q, self.s)]

    def io(self):
        return (self.X,), (self.q, self.s)

    def describe(self):
        return {"workload": f"standalone 1x128 cast of a {self.R}x{self.C} BF16 N(0,1) tensor",
                "rows": self.R, "cols": self.C}


def time_step(args, step, fp8bs, torch, dist, local, flush, stream):
    """Warm-up, graph capture and K timed steps of one workload, then K more
    steps launched kernel by kernel with an event after each (the kernels
    table). Returns the step times, per-kernel times, clocks and launch mode."""
    launches = step.launches()

    def run_seq():
        for f in launches:
            f()

    for _ in range(args.warmup):
        run_seq()
    torch.cuda.synchronize()
    if fp8bs.fp8bs_device_status(reset=True) != 0:
        raise RuntimeError("device status error during warm-up")
    # The timed steps replay one CUDA graph of the step (the same kernels,
    # without per-launch host overhead); the dense step's graph runs its two
    # independent pairs on two streams.
    run_step, launch_mode = run_seq, "stream launches"
    if not args.no_graph:
        dag = getattr(step, "run_dag", run_seq)
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                dag()
            torch.cuda.synchronize()
            for _ in range(2):
                graph.replay()
            torch.cuda.synchronize()
            run_step = graph.replay
            launch_mode = getattr(step, "dag_desc", "CUDA graph")
        except Exception as ex:   # capture unsupported: time the stream launches
            launch_mode = f"stream launches (graph capture failed: {type(ex).__name__})"
        if fp8bs.fp8bs_device_status(reset=True) != 0:
            raise RuntimeError("device status error during graph warm-up")

    nk = len(launches)
    # Timed region: exactly K steps with CUDA events at the step boundaries
    # only (an event between two kernels costs a few microseconds on this
    # GPU, ~25 us over the dense step's seven kernels).
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    clocks = ClockSampler(smi_gpu_id(local))
    barrier(dist, local)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for s in range(args.steps):
        flush.fill_(s & 0xFF)                      # L2 flush, outside the step's events
        sev[s][0].record(stream)
        run_step()
        sev[s][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(dist, local)
    status = fp8bs.fp8bs_device_status(reset=True)
    if status != 0:
        raise RuntimeError(f"device status {status} during the timed steps")
    step_ms = [a.elapsed_time(b) for a, b in sev]

    # Per-kernel breakdown (kernels table, roofline): K more steps with an
    # event after every kernel; each kernel's time includes one event's cost.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    for s in range(args.steps):
        flush.fill_(s & 0xFF)
        ev[s][0].record(stream)
        for i, f in enumerate(launches):
            f()
            ev[s][i + 1].record(stream)
    torch.cuda.synchronize()
    if fp8bs.fp8bs_device_status(reset=True) != 0:
        raise RuntimeError("device status error during the breakdown steps")
    kern_ms = {step.names[i]: [ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps)]
               for i in range(nk)}
    return {"step_ms": step_ms, "kern_ms": kern_ms, "clocks": clk, "launch_mode": launch_mode,
            "kernels_per_step": getattr(step, "kernels_per_step", nk)}


def summarize(step, t, total_s, steps, world):
    """Throughput, kernels table, roofline of the dominant kernel and the
    casts' aggregate bandwidth of one timed workload."""
    flops, kbytes = step.work()
    kern_ms = t["kern_ms"]
    peaks, peak_src = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    hbm_peak = peaks["hbm_gbs"]
    kernels = {}
    breakdown_ms = sum(sum(ts) for ts in kern_ms.values())
    for name, ts in kern_ms.items():
        avg = sum(ts) / len(ts)
        d = {"ms": round(avg, 5), "share": round(sum(ts) / breakdown_ms, 4)}
        if name in flops:
            tf = flops[name] / (avg * 1e-3) / 1e12
            d.update(tflops=round(tf, 1), frac_fp8_peak=round(tf / fp8_peak, 4))
        else:
            gbs = kbytes[name] / (avg * 1e-3) / 1e9
            d.update(gbs=round(gbs, 1), frac_hbm=round(gbs / hbm_peak, 4))
        kernels[name] = d
    dom = max(kern_ms, key=lambda n: sum(kern_ms[n]))
    dom_avg = sum(kern_ms[dom]) / len(kern_ms[dom])
    traffic = load_traffic(dom)
    if dom in flops:
        ach = flops[dom] / (dom_avg * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(ach, 1), "peak": round(fp8_peak, 1),
                "unit": "TFLOP/s", "frac": round(ach / fp8_peak, 4), "traffic": traffic,
                "peak_source": f"{peak_src} bf16 burst x {FP8_OVER_BF16:g} (nominal fp8/bf16 ratio)"}
    else:
        ach = kbytes[dom] / (dom_avg * 1e-3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(ach / hbm_peak, 4), "traffic": traffic,
                "peak_source": peak_src}
    out = {"ms_per_step": round(total_s * 1e3 / steps, 5)}
    step_flops = sum(flops.values())
    if step_flops > 0:
        value = whole_job_throughput(step_flops * steps, world, total_s) / 1e12
        out.update(value=round(value, 2), unit=UNIT, gemm_frac_fp8_peak=round(value / fp8_peak, 4))
    else:   # a cast-only workload: bandwidth
        gbs = whole_job_throughput(sum(kbytes.values()) * steps, world, total_s) / 1e9
        out.update(value=round(gbs, 1), unit="GB/s", frac_hbm=round(gbs / hbm_peak, 4))
    quant_names = [n for n in step.names if n not in flops]
    if quant_names:
        q_bytes = sum(kbytes[n] for n in quant_names)
        q_ms = sum(sum(kern_ms[n]) for n in quant_names) / steps
        out["quantize_gbs"] = round(q_bytes / (q_ms * 1e-3) / 1e9, 1)
        out["quantize_frac_hbm"] = round(q_bytes / (q_ms * 1e-3) / 1e9 / hbm_peak, 4)
    out.update(roofline=roof, kernels=kernels)
    return out


DATA = {"dense": "synthetic (seeded normal; 0.1% outliers in X)",
        "moe": "synthetic (seeded normal; Dirichlet(0.5) expert counts)",
        "longk": "synthetic (seeded uniform U(0.5, 1.5))",
        "quant16k": "synthetic (seeded normal)",
        "dense_ue8m0": "synthetic (seeded normal; 0.1% outliers in X)",
        "moe_ue8m0": "synthetic (seeded normal; Dirichlet(0.5) expert counts)"}


def make_workload(name, fp8bs, torch, device, rank):
    M, K, N = dense_shapes().values()
    if name == "moe":
        return MoeStep(fp8bs, torch, device, seed=rank)
    if name == "longk":
        return LongKStep(fp8bs, torch, device, seed=rank)
    if name == "quant16k":
        return Quant1x128Step(fp8bs, torch, device, seed=rank)
    if name == "dense_ue8m0":
        return DenseUe8m0Step(fp8bs, torch, device, M, K, N, seed=rank)
    if name == "moe_ue8m0":
        return MoeUe8m0Step(fp8bs, torch, device, seed=rank)
    return DenseStep(fp8bs, torch, device, M, K, N, seed=rank)


# Workloads the default run times after the dense step, each reported under
# its own key of "configs": the grouped MoE pass (fp32 scales with software
# promotion, and power-of-two scales on the tensor core's block scaling), the
# long-K sweep and the standalone 16384 x 16384 1x128 cast.
EXTRA_WORKLOADS = ("dense_ue8m0", "moe", "moe_ue8m0", "longk", "quant16k")


def run_ours(args, world, rank, local):
    import torch
    import fp8_block_scaled_act_gb300 as fp8bs

    fp8bs.build()
    fp8bs.lib()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    M, K, N = dense_shapes().values()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()

    def make_step():
        return make_workload(args.workload, fp8bs, torch, device, rank)

    step = make_step()
    t = time_step(args, step, fp8bs, torch, dist, local, flush, stream)
    total_s = max_over_ranks(dist, sum(t["step_ms"]) / 1e3, device=device)
    summ = summarize(step, t, total_s, args.steps, world)
    flops, _ = step.work()
    step_flops = sum(flops.values())
    e2e = None
    if step_flops > 0:
        e2e = measure_e2e(args, fp8bs, torch, [step, make_step(), make_step()], device, step_flops, world,
                          dist)

    line = {
        "metric": METRIC, "value": summ["value"], "unit": summ["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": summ["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": DATA[args.workload],
        "config": dict(step.describe(),
                       parallelism=f"replicas x{world}" if world > 1 else "1 GPU",
                       l2="flushed between steps (256 MiB write outside the step events)",
                       launch=t["launch_mode"]),
    }
    for k in ("quantize_gbs", "quantize_frac_hbm", "gemm_frac_fp8_peak", "frac_hbm", "roofline", "kernels"):
        if k in summ:
            line[k] = summ[k]
    line["kernels_note"] = ("per-kernel times from a second pass of the same K steps launched one kernel at a "
                            "time on one stream with an event after every kernel (each includes one event's "
                            "cost, a few us); ms_per_step and value come from the timed steps with events at "
                            "step boundaries only")
    if e2e is not None:
        line["e2e"] = e2e
    line["gpu_launches"] = t["kernels_per_step"] * args.steps
    line["clocks"] = t["clocks"]
    del step
    if args.workload == "dense" and not args.dense_only:
        # the other configurations of the path, each timed the same way
        configs = {}
        for name in EXTRA_WORKLOADS:
            st = make_workload(name, fp8bs, torch, device, rank)
            te = time_step(args, st, fp8bs, torch, dist, local, flush, stream)
            ts = max_over_ranks(dist, sum(te["step_ms"]) / 1e3, device=device)
            c = {"config": st.describe(), "data": DATA[name], "launch": te["launch_mode"]}
            c.update(summarize(st, te, ts, args.steps, world))
            c["gpu_launches"] = te["kernels_per_step"] * args.steps
            c["clocks"] = te["clocks"]
            configs[name] = c
            del st
            torch.cuda.empty_cache()
        line["configs"] = configs
    if rank == 0:
        if args.workload == "dense":
            line["cpu_baseline"] = cpu_baseline(M, K, N, args.cpu_baseline_sample)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def load_traffic(kernel_name):
    """DRAM bytes per launch of `kernel_name` from the committed ncu summary,
    if one exists for the current sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    return t.get(kernel_name)


def _cpulist(text):
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        lo, _, hi = part.partition("-")
        cpus.update(range(int(lo), int(hi or lo) + 1))
    return cpus


def gpu_local_cpus(torch, device):
    """(NUMA node, CPUs of that node) of the host memory nearest the GPU, from
    sysfs; (None, None) where the system does not say."""
    try:
        pr = torch.cuda.get_device_properties(device)
        addr = f"{pr.pci_domain_id:04x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0"
        with open(f"/sys/bus/pci/devices/{addr}/numa_node") as f:
            node = int(f.read())
        if node < 0:
            return None, None
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            return node, _cpulist(f.read())
    except (AttributeError, OSError, RuntimeError, ValueError):
        return None, None


def alloc_pinned_near_gpu(torch, device, make):
    """Runs `make` (which allocates the pinned host buffers) with this process
    restricted to the CPUs of the GPU's NUMA node, so that first touch puts
    the buffers in the host memory nearest the GPU; the affinity is restored
    afterwards. Returns (make's result, a note on the placement)."""
    node, cpus = gpu_local_cpus(torch, device)
    allowed = os.sched_getaffinity(0)
    use = (cpus or set()) & allowed
    note = {"gpu_numa_node": node, "bound_cpus": len(use) if use else 0}
    if not use:
        return make(), note
    os.sched_setaffinity(0, use)
    try:
        return make(), note
    finally:
        os.sched_setaffinity(0, allowed)


def measure_e2e(args, fp8bs, torch, steps, device, step_flops, world, dist):
    """Same step through the public API with host buffers: every step copies
    its inputs in from pinned host memory, runs, and copies its outputs
    (Y, dX, dW) back. Consecutive steps are pipelined on three streams over
    len(steps) sets of device tensors (step objects, three here): step i's
    input copy starts once step i - len(steps) has copied its outputs out,
    so the host link carries both directions while the kernels run, as a
    data pipeline would run it."""
    def make():
        h_in = [t.cpu().pin_memory() for t in steps[0].io()[0]]
        h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in st.io()[1]] for st in steps]
        return h_in, h_out

    (h_in, h_out), placement = alloc_pinned_near_gpu(torch, device, make)
    launches = [st.launches() for st in steps]
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    nbuf = len(steps)
    free = [None] * nbuf

    def run(n, start=None):
        for i in range(n):
            b = i % nbuf
            d_in, d_out = steps[b].io()
            if free[b] is not None:
                h2d.wait_event(free[b])
            with torch.cuda.stream(h2d):
                if i == 0 and start is not None:
                    start.record(h2d)
                for h, d in zip(h_in, d_in):
                    d.copy_(h, non_blocking=True)
            arrived = torch.cuda.Event()
            arrived.record(h2d)
            comp.wait_event(arrived)
            for f in launches[b]:
                f()
            done = torch.cuda.Event()
            done.record(comp)
            d2h.wait_event(done)
            with torch.cuda.stream(d2h):
                for h, d in zip(h_out[b], d_out):
                    h.copy_(d, non_blocking=True)
            free[b] = torch.cuda.Event()
            free[b].record(d2h)

    run(max(nbuf, args.warmup))
    torch.cuda.synchronize()
    free = [None] * nbuf
    n = max(1, args.steps)
    barrier(dist, device.index)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    run(n, start=s)
    e.record(d2h)
    torch.cuda.synchronize()
    sec = max_over_ranks(dist, s.elapsed_time(e) / 1e3, device=device)
    h2d_b = sum(t.numel() * t.element_size() for t in h_in)
    d2h_b = sum(t.numel() * t.element_size() for t in h_out[0])
    return {"value": round(whole_job_throughput(step_flops * n, world, sec) / 1e12, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
            "ms_per_step": round(sec * 1e3 / n, 4),
            "pipeline": f"host copies overlap the kernels of neighbouring steps (three streams, {nbuf} device "
                        "buffer sets)",
            "host_buffers": placement}


# ---------------------------------------------------------------------------
# the oracle as CPU baseline / reference arm
# ---------------------------------------------------------------------------

def oracle_step_sample(M, K, N, frac_rows, seed=0):
    """The dense step on the CPU oracle, restricted to a leading fraction of
    the rows of every output (and of every quantizer input). Returns
    (seconds, fraction of the full step's work it covers, cores)."""
    import numpy as np
    import oracle
    import workloads as wl

    m = max(128, int(M * frac_rows) // 128 * 128)
    nrows_w = max(128, int(N * frac_rows) // 128 * 128)
    d = wl.backward(M=m, K=K, N=N, seed=seed)
    x, w, dy = wl.bits(d["X"]), wl.bits(d["W"]), wl.bits(d["dY"])
    t0 = time.perf_counter()
    wq, sw = oracle.quant_128x128(w)
    xq, sx = oracle.quant_1x128(x)
    oracle.fprop(xq, sx, wq, sw)
    dyq, sdy = oracle.quant_1x128(dy)
    oracle.dgrad(dyq, sdy, wq, sw)
    xT, sxT = oracle.requant_128x1_T(xq, sx)
    dyT, sdyT = oracle.requant_128x1_T(dy)
    # Wgrad: rows [0, nrows_w) of dW over the m sampled tokens
    nn = np.repeat(np.arange(nrows_w), K)
    kk = np.tile(np.arange(K), nrows_w)
    oracle.wgrad(dyT, sdyT, xT, sxT, nn, kk)
    sec = time.perf_counter() - t0
    # fraction of the full step's GEMM work done (the quantizers scale alike)
    work_full = 3.0 * M * N * K
    work_done = 2.0 * m * N * K + nrows_w * K * m
    return sec, work_done / work_full, oracle.num_threads(), m, nrows_w


def cpu_baseline(M, K, N, frac):
    import oracle
    oracle.build()
    sec, covered, cores, m, nw = oracle_step_sample(M, K, N, frac)
    flops = 3 * 2.0 * M * N * K * covered
    return {"value": round(flops / sec / 1e12, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"dense step on {m} of {M} token rows (all quantizers and Fprop/Dgrad), "
                       f"Wgrad rows [0,{nw}) of dW over those tokens; {covered:.4f} of the step's "
                       f"GEMM work in {sec:.2f} s; throughput = covered FLOPs / wall time")}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    M, K, N = dense_shapes().values()
    for _ in range(args.warmup):
        oracle_step_sample(M, K, N, args.cpu_sample)
    secs, covs = [], []
    cores = 1
    for s in range(args.steps):
        sec, cov, cores, m, nw = oracle_step_sample(M, K, N, args.cpu_sample, seed=s)
        secs.append(sec)
        covs.append(cov)
    flops = sum(3 * 2.0 * M * N * K * c for c in covs)
    value = flops / sum(secs) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sum(secs) * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": f"dense FP8 linear fwd+bwd X {M}x{K}, W {K}x{N}, dY {M}x{N}",
                   "M": M, "K": K, "N": N, "parallelism": "CPU oracle on rank 0"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: the dense step on {m} of {M} token rows and "
                                   f"{nw} rows of dW ({covs[0]:.4f} of the GEMM work)"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


NCU_CASES = ("fprop", "dgrad", "wgrad", "quant_1x128", "quant_128x128", "requant_e4m3",
             "requant_bf16", "fprop_dense", "dgrad_dense", "wgrad_dense", "quant_dual", "quant_sr",
             "mx_quant", "mx_gemm", "splitk_longk", "quant_dual_stash")


def run_ncu_case(name):
    """One kernel kind, launched three times on a small case for ncu (inputs
    larger than L2, well under a few GB on the device)."""
    import torch
    import fp8_block_scaled_act_gb300 as e
    e.build()
    e.lib()
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    bf = torch.bfloat16

    def rnd(*shape, std=1.0):
        return (torch.randn(*shape, device=dev, generator=g) * std).to(bf)

    M, K, N = 16384, 7168, 2048
    if name == "fprop":
        xq, sx = e.empty_quant_1x128(M, K)
        e.fp8_quant_1x128(rnd(M, K), xq, sx)
        wq, _, sw = e.empty_quant_128x128(K, N, with_transpose=False)
        e.fp8_quant_128x128(rnd(K, N, std=0.02), wq, None, sw)
        y = torch.empty(M, N, dtype=bf, device=dev)
        runs = lambda: e.fp8_block_gemm_fprop_wkn(xq, sx, wq, sw, y)
    elif name == "dgrad":
        dyq, sdy = e.empty_quant_1x128(M, N)
        e.fp8_quant_1x128(rnd(M, N, std=1e-3), dyq, sdy)
        wq, wqT, sw = e.empty_quant_128x128(K, N)
        e.fp8_quant_128x128(rnd(K, N, std=0.02), wq, wqT, sw)
        dx = torch.empty(M, K, dtype=bf, device=dev)
        runs = lambda: e.fp8_block_gemm_dgrad(dyq, sdy, wq, sw, dx)
    elif name == "wgrad":
        xT, sxT = e.empty_requant_128x1_T(M, K)
        e.fp8_requant_128x1_T(rnd(M, K), None, xT, sxT)
        dyT, sdyT = e.empty_requant_128x1_T(M, N)
        e.fp8_requant_128x1_T(rnd(M, N, std=1e-3), None, dyT, sdyT)
        dw = torch.empty(N, K, dtype=torch.float32, device=dev)
        runs = lambda: e.fp8_block_gemm_wgrad(dyT, sdyT, xT, sxT, dw)
    elif name == "quant_1x128":
        x = rnd(16384, 16384)
        q, s = e.empty_quant_1x128(16384, 16384)
        runs = lambda: e.fp8_quant_1x128(x, q, s)
    elif name == "quant_128x128":
        w = rnd(32, 2048, 7168, std=0.02)
        q, _, s = e.empty_quant_128x128(2048, 7168, batch=32, with_transpose=False)
        runs = lambda: e.fp8_quant_128x128(w, q, None, s)
    elif name == "requant_e4m3":
        xq, sx = e.empty_quant_1x128(M, K)
        e.fp8_quant_1x128(rnd(M, K), xq, sx)
        xT, sxT = e.empty_requant_128x1_T(M, K)
        runs = lambda: e.fp8_requant_128x1_T(xq, sx, xT, sxT)
    elif name == "requant_bf16":
        x = rnd(M, K)
        xT, sxT = e.empty_requant_128x1_T(M, K)
        runs = lambda: e.fp8_requant_128x1_T(x, None, xT, sxT)
    elif name in ("fprop_dense", "dgrad_dense", "wgrad_dense"):
        # the dense bench workload's shapes exactly (for per-launch DRAM traffic)
        Md, Kd, Nd = dense_shapes().values()
        if name == "fprop_dense":
            xq, sx = e.empty_quant_1x128(Md, Kd)
            e.fp8_quant_1x128(rnd(Md, Kd), xq, sx)
            wq, _, sw = e.empty_quant_128x128(Kd, Nd, with_transpose=False)
            e.fp8_quant_128x128(rnd(Kd, Nd, std=0.02), wq, None, sw)
            y = torch.empty(Md, Nd, dtype=bf, device=dev)
            runs = lambda: e.fp8_block_gemm_fprop_wkn(xq, sx, wq, sw, y)
        elif name == "dgrad_dense":
            dyq, sdy = e.empty_quant_1x128(Md, Nd)
            e.fp8_quant_1x128(rnd(Md, Nd, std=1e-3), dyq, sdy)
            wq, wqT, sw = e.empty_quant_128x128(Kd, Nd)
            e.fp8_quant_128x128(rnd(Kd, Nd, std=0.02), wq, wqT, sw)
            dx = torch.empty(Md, Kd, dtype=bf, device=dev)
            runs = lambda: e.fp8_block_gemm_dgrad(dyq, sdy, wq, sw, dx)
        else:
            xq, sx = e.empty_quant_1x128(Md, Kd)
            e.fp8_quant_1x128(rnd(Md, Kd), xq, sx)
            xT, sxT = e.empty_requant_128x1_T(Md, Kd)
            e.fp8_requant_128x1_T(xq, sx, xT, sxT)
            dyT, sdyT = e.empty_requant_128x1_T(Md, Nd)
            e.fp8_requant_128x1_T(rnd(Md, Nd, std=1e-3), None, dyT, sdyT)
            dw = torch.empty(Nd, Kd, dtype=torch.float32, device=dev)
            runs = lambda: e.fp8_block_gemm_wgrad(dyT, sdyT, xT, sxT, dw)
    elif name == "quant_dual":
        x = rnd(M, K, std=1e-3)
        q, s = e.empty_quant_1x128(M, K)
        qT, sT = e.empty_requant_128x1_T(M, K)
        runs = lambda: e.fp8_quant_dual(x, q, s, qT, sT)
    elif name == "quant_dual_stash":
        x = rnd(M, K)
        q, s = e.empty_quant_1x128(M, K)
        qT, sT = e.empty_requant_128x1_T(M, K)
        runs = lambda: e.fp8_quant_dual_stash(x, q, s, qT, sT)
    elif name == "quant_sr":
        x = rnd(M, K)
        q, s = e.empty_quant_1x128(M, K)
        runs = lambda: e.fp8_quant_1x128_sr(x, q, s, seed=1, salt=2)
    elif name == "mx_quant":
        x = rnd(M, K)
        q, at = e.empty_mx_quant(M, K)
        runs = lambda: e.fp8_mx_quant_1x32(x, q, at)
    elif name == "mx_gemm":
        qa, aa = e.empty_mx_quant(M, K)
        e.fp8_mx_quant_1x32(rnd(M, K), qa, aa)
        qb, ab = e.empty_mx_quant(N, K)
        e.fp8_mx_quant_1x32(rnd(N, K, std=0.02), qb, ab)
        y = torch.empty(M, N, dtype=bf, device=dev)
        runs = lambda: e.fp8_mx_gemm(qa, aa, qb, ab, y)
    else:   # splitk_longk: 256 x 65536 x 256, default split
        Kl = 65536
        xq, sx = e.empty_quant_1x128(256, Kl)
        e.fp8_quant_1x128(rnd(256, Kl), xq, sx)
        wq, _, sw = e.empty_quant_128x128(Kl, 256, with_transpose=False)
        e.fp8_quant_128x128(rnd(Kl, 256, std=0.02), wq, None, sw)
        y = torch.empty(256, 256, dtype=bf, device=dev)
        op = e.OP_FPROP_WKN
        sp = e.fp8bs_splitk_default_splits(op, 256, 256, Kl)
        ws = torch.empty(e.fp8bs_splitk_workspace_size(op, 256, 256, Kl, sp), dtype=torch.uint8, device=dev)
        runs = lambda: e.fp8_block_gemm_splitk(op, xq, sx, wq, sw, y, splits=sp, workspace=ws)
    for _ in range(3):
        runs()
    torch.cuda.synchronize()
    if e.fp8bs_device_status(reset=True) != 0:
        raise RuntimeError("device status error")
    print(f"ncu case {name}: ok")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the step as stream launches instead of one CUDA graph replay")
    ap.add_argument("--dense-only", action="store_true",
                    help="time only the dense step (skip the MoE, long-K and 16384^2 cast configs)")
    ap.add_argument("--workload", choices=["dense", "moe", "longk", "quant16k", "dense_ue8m0", "moe_ue8m0"],
                    default="dense",
                    help="dense: the linear layer's fwd+bwd (default); moe: grouped expert pass; "
                         "longk: 256xKx256 split-K Fprop for K up to 65536; dense_ue8m0 / moe_ue8m0: the dense "
                         "step / expert pass with power-of-two scales, GEMMs on the tensor core's block scaling")
    ap.add_argument("--cpu-sample", type=float, default=1.0 / 16,
                    help="--impl reference: fraction of token rows the oracle runs per step")
    ap.add_argument("--cpu-baseline-sample", type=float, default=1.0,
                    help="fraction of token rows of the one oracle step timed for cpu_baseline "
                         "(1.0: the whole dense step, about 15 s on 16 host cores)")
    ap.add_argument("--ncu-case", choices=NCU_CASES, default=None,
                    help="run one kernel kind three times on a small case (for ncu) and exit")
    args = ap.parse_args(argv)
    if args.ncu_case:
        run_ncu_case(args.ncu_case)
        return
    if args.impl == "ours":
        args.warmup = max(args.warmup, 3)     # timing rule: at least 3 warm-up steps
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
