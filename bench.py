"""Benchmark: causal attention by the Ring-Attention schedule on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...      (the fp64 CPU oracle, timed)

One step = one full ring forward over the sequence (all P virtual-rank steps)
through cp_ring_forward, on inputs already resident in HBM: for bf16 rings
all steps run in one launch (each query tile walks its rank's held KV chunks
in step order and merges on chip); the _steps workloads run one launch per
step with the LSE merge in the attention epilogue.  Prints ONE JSON line on rank 0.

Workloads (synthetic, seeded N(0,1) inputs, the handbook's make_qkv recipe):
  ring128k_zigzag (default)  S=131072 H=32 D=128 bf16, P=8 zigzag
  ring128k_contiguous        same, contiguous layout
  ring128k_striped           same, striped layout (rank r holds tokens r, r+8, ...)
  ring128k_zigzag_copy       same as the default, KV physically passed to rank+1 through
                             double buffers on a second stream (copy-mode ring)
  ring32k_zigzag             S=32768, P=8 zigzag
  ring4k_zigzag              S=4096, P=4 zigzag
  ring*_zigzag_steps         the same rings, one launch per step (cp_ring_forward_steps)
  ulysses64k                 S=65536, 32 q / 8 kv heads, P=8 Ulysses
  usp64k                     the same shapes, Ulysses over 4 head groups x zigzag ring of 2
  lse_merge128k              the stand-alone LSE merge over S=131072, H=32, D=128 fp32 (GB/s)
  permute64k                 Ulysses seq_to_head of q, k, v and head_to_seq of out at the
                             ulysses64k shapes (GB/s)

FLOPs are the causal ones: 4 D H per visible (query, key) pair, i.e.
2 D H S (S + 1) per forward (the "2 S^2 H D" convention up to 1/S).
"""

import argparse
import contextlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal attention TFLOP/s & tokens/s at S=32K–128K bf16; % of GB300 bf16 peak"

WORKLOADS = {
    "ring128k_zigzag": dict(kind="ring", S=131072, H=32, Hkv=32, D=128, P=8, layout="zigzag"),
    "ring128k_contiguous": dict(kind="ring", S=131072, H=32, Hkv=32, D=128, P=8,
                                layout="contiguous"),
    "ring128k_striped": dict(kind="ring", S=131072, H=32, Hkv=32, D=128, P=8, layout="striped"),
    "ring128k_zigzag_copy": dict(kind="ring_copy", S=131072, H=32, Hkv=32, D=128, P=8,
                                 layout="zigzag"),
    "ring32k_zigzag": dict(kind="ring", S=32768, H=32, Hkv=32, D=128, P=8, layout="zigzag"),
    "ring4k_zigzag": dict(kind="ring", S=4096, H=32, Hkv=32, D=128, P=4, layout="zigzag"),
    # the same rings as one launch per step, merging through the accumulator
    "ring128k_zigzag_steps": dict(kind="ring_steps", S=131072, H=32, Hkv=32, D=128, P=8,
                                  layout="zigzag"),
    "ring32k_zigzag_steps": dict(kind="ring_steps", S=32768, H=32, Hkv=32, D=128, P=8,
                                 layout="zigzag"),
    "ring4k_zigzag_steps": dict(kind="ring_steps", S=4096, H=32, Hkv=32, D=128, P=4,
                                layout="zigzag"),
    "ulysses64k": dict(kind="ulysses", S=65536, H=32, Hkv=8, D=128, P=8, layout="ulysses"),
    "usp64k": dict(kind="usp", S=65536, H=32, Hkv=8, D=128, P=8, Pu=4, Pr=2, layout="zigzag"),
    # backward (gradients of the ring forward) and a training step (forward + backward)
    "ring128k_zigzag_bwd": dict(kind="ring_bwd", S=131072, H=32, Hkv=32, D=128, P=8,
                                layout="zigzag"),
    "ring32k_zigzag_bwd": dict(kind="ring_bwd", S=32768, H=32, Hkv=32, D=128, P=8,
                               layout="zigzag"),
    "ring128k_zigzag_train": dict(kind="ring_train", S=131072, H=32, Hkv=32, D=128, P=8,
                                  layout="zigzag"),
    # HBM-bound kernels on their own
    "lse_merge128k": dict(kind="merge", S=131072, H=32, Hkv=32, D=128, P=8, layout="-"),
    "permute64k": dict(kind="permute", S=65536, H=32, Hkv=8, D=128, P=8, layout="ulysses"),
}


def causal_flops(S, H, D):
    return 2.0 * D * H * S * (S + 1)


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value, world):
    """Max of a float over ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


FWD_KERNEL_SOURCES = ("attn_tc.cu", "attn_fwd_common.cuh", "sm100.cuh", "internal.h")


def forward_kernel_sha():
    """Digest of the sources the forward attention kernel is compiled from."""
    import hashlib
    h = hashlib.sha256()
    for name in FWD_KERNEL_SOURCES:
        with open(os.path.join(ROOT, "context_causal_attention_attn_gb300", "csrc", name),
                  "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(workload):
    """Per-launch DRAM bytes of the attention kernel from the committed ncu
    summary, or None when absent or taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "attn_fwd_tc_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_sha") != forward_kernel_sha():
        return None
    return d.get("per_launch_bytes", {}).get(workload)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------- host buffers and the link
def gpu_numa_node(local):
    """NUMA node of the GPU's PCI function as the kernel reports it, or None."""
    bus = None
    try:
        import torch
        p = torch.cuda.get_device_properties(local)
        bus = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(local), "--query-gpu=pci.bus_id",
                                  "--format=csv,noheader"], capture_output=True, text=True,
                                 timeout=30).stdout.strip()
            dom, rest = out.split(":", 1)
            bus = f"{int(dom, 16):04x}:{rest.lower()}"
        except Exception:
            return None
    try:
        with open(f"/sys/bus/pci/devices/{bus}/numa_node") as f:
            node = int(f.read().strip())
    except Exception:
        return None
    return node if node >= 0 else None


def _node_cpus(node):
    cpus = set()
    try:
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            for part in f.read().strip().split(","):
                if "-" in part:
                    a, b = part.split("-")
                    cpus.update(range(int(a), int(b) + 1))
                elif part:
                    cpus.add(int(part))
    except Exception:
        pass
    return cpus


@contextlib.contextmanager
def near_gpu(local):
    """Narrow this process's CPU affinity to the GPU's NUMA node while
    page-locked host buffers are allocated (pages are placed on the node of
    the CPU that first touches them), then restore it.  Yields the node, or
    None when the platform does not say or no allowed CPU is on it."""
    node = gpu_numa_node(local)
    old = os.sched_getaffinity(0)
    cpus = (_node_cpus(node) & old) if node is not None else set()
    if cpus:
        os.sched_setaffinity(0, cpus)
    try:
        yield node if cpus else None
    finally:
        if cpus:
            os.sched_setaffinity(0, old)


def link_gbs(dev_t, host_t, stream, samples=5):
    """Host-to-device and device-to-host GB/s of plain copies between a
    page-locked host tensor and a device tensor of the same size, each copy
    timed alone with CUDA events on ``stream``.  Returns (median H2D, median
    D2H, bytes, {"h2d": [min, max], "d2h": [min, max]}): the host link of a
    shared machine can slow down for seconds at a time, which the spread
    shows."""
    import torch
    nbytes = dev_t.numel() * dev_t.element_size()
    med, spread = [], {}
    for h2d in (True, False):
        dst, src = (dev_t, host_t) if h2d else (host_t, dev_t)
        dst.copy_(src, non_blocking=True)
        rates = []
        for _ in range(samples):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(src, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            rates.append(nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
        med.append(round(statistics.median(rates), 1))
        spread["h2d" if h2d else "d2h"] = [round(min(rates), 1), round(max(rates), 1)]
    return med[0], med[1], nbytes, spread


def l2_cache_bytes(dev):
    import torch
    props = torch.cuda.get_device_properties(dev)
    return int(getattr(props, "L2_cache_size", 0) or (128 << 20))


def timed_calls(fn, n, stream):
    """Run fn n times back to back with an event between calls; returns
    (total ms, [ms per call])."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    evs[0].record(stream)
    for i in range(n):
        fn()
        evs[i + 1].record(stream)
    evs[n].synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]
    return evs[0].elapsed_time(evs[n]), per


def timed_steps(step, K, min_timed_s, stream):
    """Steps to time: at least K, and enough to fill ``min_timed_s`` seconds
    so that the 200 ms clock sampler sees the timed region (short workloads
    run in milliseconds).  One extra untimed step measures the step time."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    step()
    e1.record(stream)
    e1.synchronize()
    ms = max(e0.elapsed_time(e1), 1e-3)
    return max(K, int(math.ceil(min_timed_s * 1e3 / ms)))


# --------------------------------------------------------------- CPU oracle
def host_inputs(wl, seed=0, device_tensors=None):
    """float32 host copies of the workload's bf16 q, k, v (exact widening)."""
    import torch

    from context_causal_attention_attn_gb300.inputs import make_qkv
    if device_tensors is None:
        device_tensors = make_qkv(wl["S"], wl["H"], wl["D"], Hkv=wl["Hkv"],
                                  dtype=torch.bfloat16, seed=seed)
    return [t.float().cpu().numpy() for t in device_tensors]


ORACLE_ROWS_PER_CALL = 64


def cpu_oracle_sample(wl, qkv, budget_s=15.0, seed=0, max_calls=None):
    """Time the fp64 oracle on a bounded sample of the workload: calls of
    ORACLE_ROWS_PER_CALL seeded query rows (all heads) against every key they
    see, repeated until the time budget is spent (or ``max_calls`` calls).
    Every call has the same size, so the cpu_baseline leg (several calls)
    and each step of the reference arm (one call) time the same unit of work.
    Returns (TFLOP/s over the causal pairs evaluated, description, host
    cores, seconds, calls)."""
    import numpy as np

    import oracle
    from context_causal_attention_attn_gb300.inputs import sample_rows

    S, H, D = wl["S"], wl["H"], wl["D"]
    qf, kf, vf = qkv
    cores = len(os.sched_getaffinity(0))
    n = min(ORACLE_ROWS_PER_CALL, S)
    spent, flops, rows_done, calls = 0.0, 0.0, 0, 0
    while spent < budget_s and (max_calls is None or calls < max_calls):
        rows = sample_rows(S, n, seed=seed * 7919 + calls + 1)
        t0 = time.perf_counter()
        oracle.attention_monolithic(qf, kf, vf, rows=rows)
        spent += time.perf_counter() - t0
        flops += float(np.sum(4.0 * D * H * (rows + 1)))
        rows_done += len(rows)
        calls += 1
    desc = (f"{calls} call(s) of {n} seeded query rows x {H} heads of the {S}-token sequence "
            f"against every key they see ({rows_done} rows; fp64 NumPy oracle, BLAS threads = "
            f"host cores)")
    return flops / spent / 1e12, desc, cores, spent, calls


# --------------------------------------------------------------- GPU path
def per_rank_times(cp, q, k, v, P, layout, stream):
    """Load-balance indicator: every block of every ring step, run alone
    through cp_attn_block with its chunk offsets and timed with CUDA events,
    summed per virtual rank (the ring's own launches run all ranks at once,
    so they show no per-rank time).  Returns (ms per rank, max / mean)."""
    import torch
    S, H, D = q.shape
    n = 2 * P if layout == "zigzag" else P
    C = S // n
    out = torch.empty(C, H, D, dtype=torch.bfloat16, device=q.device)
    lse = torch.empty(H, C, dtype=torch.float32, device=q.device)
    blocks = [b for t in range(P) for b in cp.cp_ring_step_blocks(P, layout, t)]

    def run(r, qc, kc):
        cp.cp_attn_block(q[qc * C:(qc + 1) * C], k[kc * C:(kc + 1) * C], v[kc * C:(kc + 1) * C],
                         q_offset=qc * C, k_offset=kc * C, out=out, lse=lse, stream=stream)

    for r, qc, kc, _ in blocks[:4]:
        run(r, qc, kc)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in blocks]
    for (e0, e1), (r, qc, kc, _) in zip(evs, blocks):
        e0.record(stream)
        run(r, qc, kc)
        e1.record(stream)
    torch.cuda.synchronize(q.device)
    per = [0.0] * P
    for (e0, e1), (r, _, _, _) in zip(evs, blocks):
        per[r] += e0.elapsed_time(e1)
    return [round(x, 2) for x in per], round(max(per) / (sum(per) / P), 3)


def run_gpu(args, wl, rank, world, local):
    import torch

    import context_causal_attention_attn_gb300 as cp
    from context_causal_attention_attn_gb300 import build as cpbuild
    from context_causal_attention_attn_gb300.inputs import make_qkv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # one rank compiles (if needed); the others load the result after the barrier
    if rank == 0:
        cpbuild.build()
    barrier(world)
    cp.lib()
    S, H, Hkv, D, P, layout = wl["S"], wl["H"], wl["Hkv"], wl["D"], wl["P"], wl["layout"]
    q, k, v = make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=rank, device=dev)
    out = torch.empty(S, H, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(H, S, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ring_impl = None
    if wl["kind"] in ("ring", "ring_steps"):
        ws = torch.empty(max(cp.cp_ring_workspace_size(S, H, D, torch.bfloat16), 16),
                         dtype=torch.uint8, device=dev)
        one_launch = wl["kind"] == "ring" and cp.ring_runs_fused(q, layout)
        launches_per_step = 1 if one_launch else P
        attn_stages = set(range(launches_per_step))  # every launch is attention
        ring_fn = cp.cp_ring_forward if wl["kind"] == "ring" else cp.cp_ring_forward_steps
        ring_impl = (f"cp_ring_forward: all {P} steps in one launch (each query tile walks its "
                     "rank's held KV chunks in step order, merging on chip)" if one_launch else
                     f"{ring_fn.__name__}: one launch per step ({P}), each merging into the "
                     "fp32 accumulator in its epilogue")

        def step():
            ring_fn(q, k, v, P, layout, out=out, lse=lse, workspace=ws, stream=stream)
    elif wl["kind"] == "ring_copy":
        ws = torch.empty(cp.cp_ring_copy_workspace_size(S, H, Hkv, D, P, layout, torch.bfloat16,
                                                        torch.bfloat16), dtype=torch.uint8,
                         device=dev)
        side = torch.cuda.Stream(dev)
        launches_per_step = P  # plus the D2D copies on the side stream

        def step():
            cp.cp_ring_forward_copy(q, k, v, P, layout, out=out, lse=lse, workspace=ws,
                                    stream=stream, copy_stream=side)
    elif wl["kind"] == "usp":
        ws = torch.empty(cp.cp_usp_workspace_size(S, H, Hkv, D, torch.bfloat16, torch.bfloat16),
                         dtype=torch.uint8, device=dev)
        if cp.ring_runs_fused(q, layout):
            # the whole ring is stage 1 (one launch); stages 2..Pr launch nothing
            launches_per_step = 5  # 3 permutes, the ring, inverse permute
            stages, attn_stages = [0, 1, wl["Pr"] + 1], {1}
            ring_impl = (f"cp_usp_forward: the rings of all {wl['Pu']} head groups, all "
                         f"{wl['Pr']} steps, in one launch")
        else:
            launches_per_step = 4 + wl["Pr"]  # 3 permutes, Pr ring steps, inverse permute
            stages = list(range(wl["Pr"] + 2))  # permutes, ring steps 1..Pr, inverse permute
            attn_stages = set(range(1, wl["Pr"] + 1))

        def launch(st):
            cp.cp_usp_stage(q, k, v, wl["Pu"], wl["Pr"], layout, st, out, lse, ws, stream=stream)

        def step():
            cp.cp_usp_forward(q, k, v, wl["Pu"], wl["Pr"], layout, out=out, lse=lse, workspace=ws,
                              stream=stream)
    else:
        ws = torch.empty(cp.cp_ulysses_workspace_size(S, H, Hkv, D, torch.bfloat16,
                                                      torch.bfloat16), dtype=torch.uint8,
                         device=dev)
        launches_per_step = 5  # 3 permutes, attention, inverse permute
        stages, attn_stages = [0, 1, 2], {1}

        def launch(st):
            cp.cp_ulysses_stage(q, k, v, P, st, out, lse, ws, stream=stream)

        def step():
            cp.cp_ulysses_forward(q, k, v, P, out=out, lse=lse, workspace=ws, stream=stream)

    flops = causal_flops(S, H, D)
    for _ in range(args.warmup):
        step()
    cp.cp_check_device_error(stream)

    # timed region: per-launch events for the ring (one attention kernel per
    # ring step); whole-step events bracket everything
    K = timed_steps(step, args.steps, args.min_timed_s, stream)
    K = int(reduce_max(float(K), world))
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    per_launch = []
    barrier(world)
    torch.cuda.synchronize(dev)
    # Ulysses / USP: the step as its public stages, an event after each, so
    # that the attention launches are timed apart from the permutes.  The
    # ring runs whole cp_ring_forward calls: its steps overlap (each launch
    # starts while the previous one drains), so per-launch events would
    # change what is timed.
    staged = wl["kind"] in ("ulysses", "usp")
    # Inputs that fit in L2 (twice over) would be served from it after the
    # first step: then every timed step starts behind a write of a buffer
    # twice the size of L2, and the steps alone are timed and summed.
    l2_bytes = l2_cache_bytes(dev)
    in_bytes = sum(t.numel() * t.element_size() for t in (q, k, v))
    flush = (torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
             if in_bytes < 2 * l2_bytes else None)
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(K)] if flush is not None else []
    with ClockSampler(local) as clk:
        if staged:
            n = len(stages)
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(K)]
            ev_start.record(stream)
            for s_ in range(K):
                if flush is not None:
                    flush.fill_(s_ & 0xFF)
                evs[s_][0].record(stream)
                for i, st in enumerate(stages):
                    launch(st)
                    evs[s_][i + 1].record(stream)
            ev_end.record(stream)
        else:
            ev_start.record(stream)
            for s_ in range(K):
                if flush is not None:
                    flush.fill_(s_ & 0xFF)
                    step_evs[s_][0].record(stream)
                step()
                if flush is not None:
                    step_evs[s_][1].record(stream)
            ev_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    cp.cp_check_device_error(stream)
    if flush is None:
        total_ms = ev_start.elapsed_time(ev_end)
    elif staged:
        total_ms = sum(evs[s_][0].elapsed_time(evs[s_][len(stages)]) for s_ in range(K))
    else:
        total_ms = sum(a.elapsed_time(b) for a, b in step_evs)
    del flush
    l2_note = (f"inputs larger than L2 ({in_bytes >> 20} MiB of q/k/v per rank)"
               if not step_evs and in_bytes >= 2 * l2_bytes else
               f"L2 flushed before every timed step (a {2 * l2_bytes >> 20} MiB write; the "
               f"{in_bytes >> 20} MiB of q/k/v would fit in L2); the steps alone are timed")
    if staged:
        for s_ in range(K):
            for i, st in enumerate(stages):
                if st in attn_stages:
                    per_launch.append(evs[s_][i].elapsed_time(evs[s_][i + 1]))
    t_max_ms = reduce_max(total_ms, world)
    clocks = clk.summary()

    # end to end through the public API with pinned host buffers on the
    # GPU's NUMA node
    with near_gpu(local) as numa_node:
        hq, hk, hv = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (q, k, v))
        hout = torch.empty(S, H, D, dtype=torch.bfloat16, pin_memory=True)
        hlse = torch.empty(H, S, dtype=torch.float32, pin_memory=True)
    for h_, d_ in ((hq, q), (hk, k), (hv, v)):
        h_.copy_(d_)
    h2d_gbs, d2h_gbs, link_bytes, link_spread = link_gbs(q, hq, stream)
    q.copy_(hq)
    K_e2e = max(1, min(K, 5))
    host_api = wl["kind"] in ("ring", "ring_steps", "ulysses", "usp")
    host_fn = {"ulysses": "cp_ulysses_forward_host", "usp": "cp_usp_forward_host"}.get(
        wl["kind"], "cp_ring_forward_host")
    if wl["kind"] == "usp":
        groups = wl["Pu"]
        hws = torch.empty(cp.cp_usp_host_workspace_size(S, H, Hkv, D, wl["Pu"], torch.bfloat16,
                                                        torch.bfloat16),
                          dtype=torch.uint8, device=dev)
        side = torch.cuda.Stream(dev)
        dq = dk = dv = None
    elif wl["kind"] == "ulysses":
        # the C ABI's host-buffer Ulysses: strided copies do the all-to-alls,
        # each head group's attention overlapping the others' copies
        groups = P
        hws = torch.empty(cp.cp_ulysses_host_workspace_size(S, H, Hkv, D, P, torch.bfloat16,
                                                            torch.bfloat16),
                          dtype=torch.uint8, device=dev)
        side = torch.cuda.Stream(dev)
        dq = dk = dv = None
    elif host_api:
        # the C ABI's host-buffer entry point: copies in, ring, copies out,
        # overlapped across head groups on a second stream
        groups = max(g for g in range(1, args.host_groups + 1) if Hkv % g == 0)
        hws = torch.empty(cp.cp_ring_host_workspace_size(S, H, Hkv, D, groups, torch.bfloat16,
                                                         torch.bfloat16),
                          dtype=torch.uint8, device=dev)
        side = torch.cuda.Stream(dev)
        dq = dk = dv = None
    else:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def e2e_step():
        if wl["kind"] == "usp":
            cp.cp_usp_forward_host(hq, hk, hv, wl["Pu"], wl["Pr"], layout, hout=hout, hlse=hlse,
                                   workspace=hws, stream=stream, copy_stream=side)
            return
        if wl["kind"] == "ulysses":
            cp.cp_ulysses_forward_host(hq, hk, hv, P, hout=hout, hlse=hlse, workspace=hws,
                                       stream=stream, copy_stream=side)
            return
        if host_api:
            cp.cp_ring_forward_host(hq, hk, hv, P, layout, hout=hout, hlse=hlse, groups=groups,
                                    workspace=hws, stream=stream, copy_stream=side)
            return
        # ring_copy: pinned host copies, then the device entry point
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        cp.cp_ring_forward_copy(dq, dk, dv, P, layout, out=out, lse=lse, workspace=ws,
                                stream=stream, copy_stream=side)
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms, e2e_calls = timed_calls(e2e_step, K_e2e, stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e2e_ms, world)
    cp.cp_check_device_error(stream)
    h2d = (q.numel() + k.numel() + v.numel()) * 2
    d2h = out.numel() * 2 + lse.numel() * 4

    value = world * flops * K / (t_max_ms / 1e3) / 1e12
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "steps_requested": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max_ms / K, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v, handbook make_qkv recipe, drawn on device)",
        "config": {"workload": args.workload, "S": S, "H": H, "Hkv": Hkv, "D": D, "P": P,
                   "layout": layout, "in_dtype": "bf16", "out_dtype": "bf16",
                   "accumulate": "fp32", "causal": True,
                   "l2": l2_note,
                   "flops_per_step": flops, "parallelism": f"replicas x{world}",
                   **({"ring_impl": ring_impl} if ring_impl else {})},
        "tokens_per_s": round(world * S * K / (t_max_ms / 1e3), 1),
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"], "samples": clocks["samples"]},
        "gpu_launches": K * launches_per_step,
        "e2e": {"value": round(world * flops * K_e2e / (e2e_ms / 1e3) / 1e12, 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": K_e2e,
                "api": (host_fn + f" (pinned host buffers, {groups} head groups, copies on a "
                        "second stream)") if host_api else
                       "pinned host copies + device entry point on one stream",
                "ms_per_call": [round(x, 3) for x in e2e_calls],
                "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs, "link_gbs_min_max": link_spread,
                "link_note": (f"median of 5 plain pinned copies of q ({link_bytes >> 20} MiB) each way; "
                              f"host buffers on NUMA node {numa_node}" if numa_node is not None
                              else f"plain pinned copies of q ({link_bytes >> 20} MiB) each "
                              "way; the GPU's NUMA node is not reported, host buffers where "
                              "the allocator put them")},
    }
    peaks, peak_kind = load_peaks()
    ring_kinds = ("ring", "ring_steps", "ring_copy")
    if wl["kind"] in ring_kinds:
        # every launch on the compute stream is the attention kernel (99.8% of
        # device time in the launch list); launches run back to back (copy
        # mode: the mean includes any wait for the KV copies)
        per_launch = [total_ms / (K * launches_per_step)] * (K * launches_per_step)
        attn_stages = set(range(launches_per_step))
    if (staged or wl["kind"] in ring_kinds) and per_launch:
        mean_launch_ms = statistics.fmean(per_launch)
        achieved = flops / len(attn_stages) / (mean_launch_ms / 1e3) / 1e12
        peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
        traffic = load_traffic(args.workload)
        result["roofline"] = {
            "kernel": "attn_fwd_tc_kernel", "bound": "tensor", "achieved": round(achieved, 2),
            "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "note": (f"peak = bf16_tflops_sustained of {peak_kind} MEASURED_PEAKS (kernel timed "
                     f"inside a multi-second loop); achieved = causal FLOPs per attention "
                     f"launch (flops_per_step / {len(attn_stages)} launches per step) / mean "
                     f"launch time ({mean_launch_ms:.3f} ms over {len(per_launch)} launches; "
                     + ("the whole ring is one launch, so the mean is the step time)"
                        if wl["kind"] == "ring" and launches_per_step == 1 else
                        "the ring's launches overlap under programmatic dependent launch, so "
                        "the mean is the step time / launches)" if wl["kind"] in ring_kinds[:2] else
                        "step time / launches, including waits for the KV copies on the side "
                        "stream)" if wl["kind"] == "ring_copy" else
                        "each launch bracketed by events, permute launches excluded)"))}
    else:
        result["roofline"] = None
    if wl["kind"] in ("ring", "ring_steps") and layout in ("contiguous", "zigzag") and \
            S % (2 * P) == 0:
        per, imb = per_rank_times(cp, q, k, v, P, layout, stream)
        result["per_virtual_rank_ms"] = per
        result["virtual_rank_imbalance"] = imb
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, desc, cores, spent, _ = cpu_oracle_sample(
            wl, host_inputs(wl, device_tensors=(q, k, v)), budget_s=args.cpu_budget)
        result["cpu_baseline"] = {"value": round(val, 6), "unit": "TFLOP/s", "cores": cores,
                                  "kind": "oracle", "sample": desc,
                                  "seconds": round(spent, 1)}
    return result


def cpu_oracle_bwd_sample(wl, budget_s=15.0, seed=0, with_forward=False, max_calls=None):
    """Time the fp64 oracle backward on a bounded sample: calls of
    ORACLE_ROWS_PER_CALL seeded query rows of one head against every key they
    see (out and lse of those rows from the oracle's forward, timed only when
    with_forward), until the budget is spent or ``max_calls`` calls.  Returns
    (TFLOP/s counted as 2.5x -- 3.5x with the forward -- the causal forward
    FLOPs of the pairs evaluated, description, cores, seconds, calls)."""
    import numpy as np
    import torch

    import oracle
    from context_causal_attention_attn_gb300.inputs import make_dout, make_qkv, sample_rows

    S, H, D = wl["S"], wl["H"], wl["D"]
    q, k, v = make_qkv(S, 1, D, Hkv=1, dtype=torch.bfloat16, seed=seed)
    do = make_dout(S, 1, D, dtype=torch.bfloat16, seed=seed)
    qf, kf, vf, dof = (t.double().numpy() for t in (q, k, v, do))
    cores = len(os.sched_getaffinity(0))
    n, spent, flops, rows_done, calls = min(ORACLE_ROWS_PER_CALL, S), 0.0, 0.0, 0, 0
    while spent < budget_s and (max_calls is None or calls < max_calls):
        rows = sample_rows(S, n, seed=seed * 7919 + calls + 1)
        kmax = int(rows.max()) + 1
        t0 = time.perf_counter()
        o, l = oracle.attention(qf[rows], kf[:kmax], vf[:kmax], q_positions=rows)
        t1 = time.perf_counter()
        oracle.attention_backward(qf[rows], kf[:kmax], vf[:kmax], o, l, dof[rows],
                                  q_positions=rows)
        spent += time.perf_counter() - (t0 if with_forward else t1)
        flops += (3.5 if with_forward else 2.5) * float(np.sum(4.0 * D * (rows + 1)))
        rows_done += len(rows)
        calls += 1
    desc = (f"{'forward + ' if with_forward else ''}backward of {calls} call(s) of {n} seeded "
            f"query rows of one head of the {S}-token sequence against every key they see "
            f"({rows_done} rows; fp64 NumPy oracle, BLAS threads = host cores)")
    return flops / spent / 1e12, desc, cores, spent, calls


def run_bwd(args, wl, rank, world, local):
    """The ring backward (kind ring_bwd) or forward + backward (ring_train)
    with bf16 gradients; TFLOP/s counted on the algorithmic FLOPs (backward =
    2.5x the causal forward: the S, dP, dV, dQ, dK products)."""
    import torch

    import context_causal_attention_attn_gb300 as cp
    from context_causal_attention_attn_gb300 import build as cpbuild
    from context_causal_attention_attn_gb300.inputs import make_dout, make_qkv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # one rank compiles (if needed); the others load the result after the barrier
    if rank == 0:
        cpbuild.build()
    barrier(world)
    cp.lib()
    S, H, Hkv, D, P, layout = wl["S"], wl["H"], wl["Hkv"], wl["D"], wl["P"], wl["layout"]
    train = wl["kind"] == "ring_train"
    q, k, v = make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=rank, device=dev)
    do = make_dout(S, H, D, dtype=torch.bfloat16, seed=rank, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = torch.empty(S, H, D, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(H, S, dtype=torch.float32, device=dev)
    fws = torch.empty(max(cp.cp_ring_workspace_size(S, H, D, torch.bfloat16), 16),
                      dtype=torch.uint8, device=dev)
    cp.cp_ring_forward(q, k, v, P, layout, out=out, lse=lse, workspace=fws, stream=stream)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    bws = torch.empty(cp.cp_ring_backward_workspace_size(S, H, Hkv, D, torch.bfloat16),
                      dtype=torch.uint8, device=dev)
    # the forward of a training step: cp_ring_forward (one launch for the whole
    # ring where it runs fused, else one per step)
    fwd_launches = [("fwd", -1)] if cp.ring_runs_fused(q, layout) else [
        ("fwd", t) for t in range(P)]
    # the backward: cp_ring_backward's schedule (for bf16 inputs one dK/dV and
    # one dQ launch over every step, else one of each per step)
    fused_bwd = cp.ring_backward_runs_fused(q, layout)
    bstep = cp.cp_ring_backward_fused_step if fused_bwd else cp.cp_ring_backward_step
    nbl = 2 if fused_bwd else 2 * P
    launches = (fwd_launches if train else []) + [("delta", -1)] + [
        ("dkdv" if l % 2 == 0 else "dq", l) for l in range(nbl)]

    def launch(kind, l, tensors=(q, k, v, do)):
        q_, k_, v_, do_ = tensors
        if kind == "fwd" and l < 0:
            cp.cp_ring_forward(q_, k_, v_, P, layout, out=out, lse=lse, workspace=fws,
                               stream=stream)
        elif kind == "fwd":
            cp.cp_ring_step(q_, k_, v_, P, layout, l, out, lse, fws, stream=stream)
        else:
            bstep(q_, k_, v_, out, do_, lse, P, layout, l, dq, dk, dv, bws, stream=stream)

    def step(tensors=(q, k, v, do)):
        if train:
            cp.cp_ring_forward(tensors[0], tensors[1], tensors[2], P, layout, out=out, lse=lse,
                               workspace=fws, stream=stream)
        cp.cp_ring_backward(*tensors[:3], out, tensors[3], lse, P, layout, dq=dq, dk=dk, dv=dv,
                            workspace=bws, stream=stream)

    fwd_flops = causal_flops(S, H, D)
    flops = (3.5 if train else 2.5) * fwd_flops
    for _ in range(args.warmup):
        step()
    cp.cp_check_device_error(stream)
    K = timed_steps(step, args.steps, args.min_timed_s, stream)
    K = int(reduce_max(float(K), world))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(launches) + 1)]
           for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        for s_ in range(K):
            evs[s_][0].record(stream)
            for i, (kind, l) in enumerate(launches):
                launch(kind, l)
                evs[s_][i + 1].record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    cp.cp_check_device_error(stream)
    total_ms = evs[0][0].elapsed_time(evs[K - 1][len(launches)])
    per_kind = {}
    for s_ in range(K):
        for i, (kind, _) in enumerate(launches):
            per_kind.setdefault(kind, []).append(evs[s_][i].elapsed_time(evs[s_][i + 1]))
    t_max_ms = reduce_max(total_ms, world)
    clocks = clk.summary()

    # end to end: inputs from pinned host memory (on the GPU's NUMA node),
    # gradients back
    src = (q, k, v, do) if train else (q, k, v, do, out, lse)
    with near_gpu(local) as numa_node:
        host_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in src]
        host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
    for h_, d_ in zip(host_in, src):
        h_.copy_(d_)
    h2d_gbs, d2h_gbs, link_bytes, link_spread = link_gbs(dq, host_out[0], stream)
    K_e2e = max(1, min(K, 5))
    host_api = not train
    if host_api:
        # the C ABI's host-buffer entry point: copies in, ring backward, copies
        # out, overlapped across head groups on a second stream
        groups = max(g for g in range(1, args.host_groups + 1) if Hkv % g == 0)
        hws = torch.empty(cp.cp_ring_backward_host_workspace_size(S, H, Hkv, D, groups,
                                                                  torch.bfloat16, torch.bfloat16),
                          dtype=torch.uint8, device=dev)
        side = torch.cuda.Stream(dev)
        dev_in = []
    else:
        dev_in = [torch.empty_like(t) for t in (q, k, v, do)]

    def e2e_step():
        if host_api:
            hq_, hk_, hv_, hdo_, hout_, hlse_ = host_in
            cp.cp_ring_backward_host(hq_, hk_, hv_, hout_, hdo_, hlse_, P, layout,
                                     grad_dtype=torch.bfloat16, hdq=host_out[0],
                                     hdk=host_out[1], hdv=host_out[2], groups=groups,
                                     workspace=hws, stream=stream, copy_stream=side)
            return
        for d_, h_ in zip(dev_in, host_in):
            d_.copy_(h_, non_blocking=True)
        step(tuple(dev_in[:4]))
        for d_, h_ in zip((dq, dk, dv), host_out):
            h_.copy_(d_, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms, e2e_calls = timed_calls(e2e_step, K_e2e, stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e2e_ms, world)
    cp.cp_check_device_error(stream)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    # roofline of the kernel with the largest share: its own tensor FLOPs
    # (dK/dV kernel: S^T, dP^T, dV, dK = 2x the causal forward; dQ kernel:
    # S, dP, dQ = 1.5x; forward kernel 1x) over its launch time
    kernel_flops = {"dkdv": 2.0 * fwd_flops, "dq": 1.5 * fwd_flops, "fwd": fwd_flops}
    kernel_names = {"dkdv": "attn_bwd_tc_kernel<dK/dV>", "dq": "attn_bwd_tc_kernel<dQ>",
                    "fwd": "attn_fwd_tc_kernel"}
    shares = {kd: sum(v_) for kd, v_ in per_kind.items()}
    top = max((kd for kd in shares if kd in kernel_flops), key=lambda kd: shares[kd])
    peaks, peak_kind = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    achieved = kernel_flops[top] * K / (shares[top] / 1e3) / 1e12
    value = world * flops * K / (t_max_ms / 1e3) / 1e12
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "steps_requested": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max_ms / K, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/k/v and dO, drawn on device)",
        "config": {"workload": args.workload, "S": S, "H": H, "Hkv": Hkv, "D": D, "P": P,
                   "layout": layout, "in_dtype": "bf16", "grad_dtype": "bf16",
                   "accumulate": "fp32", "causal": True,
                   "pass": "forward + backward" if train else "backward",
                   "ring_impl": ("one dK/dV and one dQ launch over all steps (each "
                                 "stationary tile keeps its gradient on chip)" if fused_bwd else
                                 "one dK/dV and one dQ launch per step, accumulating in fp32"),
                   "l2": f"inputs larger than L2 ({h2d >> 20} MiB per rank)",
                   "flops_per_step": flops,
                   "flops_count": ("3.5x" if train else "2.5x") + " causal forward FLOPs",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(world * S * K / (t_max_ms / 1e3), 1),
        "kernel_ms_per_step": {kd: round(v_ / K, 3) for kd, v_ in shares.items()},
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"], "samples": clocks["samples"]},
        "gpu_launches": K * len(launches),
        "e2e": {"value": round(world * flops * K_e2e / (e2e_ms / 1e3) / 1e12, 2),
                "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": K_e2e,
                "api": (f"cp_ring_backward_host (pinned host buffers, {groups} head groups, "
                        "copies on a second stream)") if host_api else
                       "pinned host copies + device entry points on one stream",
                "ms_per_call": [round(x, 3) for x in e2e_calls],
                "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs, "link_gbs_min_max": link_spread,
                "link_note": (f"median of 5 plain pinned copies of {link_bytes >> 20} MiB each way; host "
                              f"buffers on NUMA node {numa_node}" if numa_node is not None else
                              f"plain pinned copies of {link_bytes >> 20} MiB each way; the "
                              "GPU's NUMA node is not reported")},
        "roofline": {
            "kernel": kernel_names[top], "bound": "tensor", "achieved": round(achieved, 2),
            "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
            "note": (f"peak = bf16_tflops_sustained of {peak_kind} MEASURED_PEAKS; achieved = "
                     f"the kernel's own products ({kernel_flops[top] / fwd_flops:.1f}x the "
                     f"causal forward FLOPs per step) / its summed launch time "
                     f"({shares[top] / K:.2f} ms per step)")},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        val, desc, cores, spent, _ = cpu_oracle_bwd_sample(wl, budget_s=args.cpu_budget,
                                                           with_forward=train)
        result["cpu_baseline"] = {"value": round(val, 6), "unit": "TFLOP/s", "cores": cores,
                                  "kind": "oracle", "sample": desc, "seconds": round(spent, 1)}
    return result


def run_hbm(args, wl, rank, world, local):
    """The HBM-bound kernels alone: bytes moved per step / time, in GB/s."""
    import torch

    import context_causal_attention_attn_gb300 as cp
    from context_causal_attention_attn_gb300 import build as cpbuild
    from context_causal_attention_attn_gb300.inputs import make_qkv

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # one rank compiles (if needed); the others load the result after the barrier
    if rank == 0:
        cpbuild.build()
    barrier(world)
    cp.lib()
    stream = torch.cuda.current_stream(dev)
    S, H, Hkv, D, P = wl["S"], wl["H"], wl["Hkv"], wl["D"], wl["P"]
    g = torch.Generator(device=dev)
    g.manual_seed(rank)
    if wl["kind"] == "merge":
        acc = torch.randn(S, H, D, generator=g, device=dev)
        blk = torch.randn(S, H, D, generator=g, device=dev)
        lacc = torch.randn(H, S, generator=g, device=dev)
        lblk = torch.randn(H, S, generator=g, device=dev)
        inputs = (acc, lacc, blk, lblk)
        # per row-head: read 2 D fp32 + 2 lse, write D fp32 + 1 lse
        algo = S * H * (3 * D * 4 + 3 * 4)
        kernel, launches = "lse_merge_kernel", 1

        def step():
            cp.cp_lse_merge(acc, lacc, blk, lblk, stream=stream)
        result_t = (acc, lacc)
    else:
        q, k, v = make_qkv(S, H, D, Hkv=Hkv, dtype=torch.bfloat16, seed=rank, device=dev)
        qh = torch.empty(P, S, H // P, D, dtype=q.dtype, device=dev)
        kh = torch.empty(P, S, Hkv // P, D, dtype=q.dtype, device=dev)
        vh = torch.empty_like(kh)
        back = torch.empty_like(q)
        inputs = (q, k, v)
        algo = 2 * (2 * q.numel() + k.numel() + v.numel()) * 2
        kernel, launches = "permute_kernel", 4

        def step():
            cp.cp_seq_to_head(q, P, qh, stream=stream)
            cp.cp_seq_to_head(k, P, kh, stream=stream)
            cp.cp_seq_to_head(v, P, vh, stream=stream)
            cp.cp_head_to_seq(qh, back, stream=stream)
        result_t = (back,)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    K = timed_steps(step, args.steps, args.min_timed_s, stream)
    K = int(reduce_max(float(K), world))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(K):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    t_ms = reduce_max(e0.elapsed_time(e1), world)
    # end to end with pinned host buffers (on the GPU's NUMA node)
    with near_gpu(local) as numa_node:
        hin = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in inputs]
        hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in result_t]
    for h_, d_ in zip(hin, inputs):
        h_.copy_(d_)
    h2d_gbs, d2h_gbs, _, link_spread = link_gbs(inputs[0], hin[0], stream)
    inputs[0].copy_(hin[0])
    K_e2e = max(1, min(K, 5))
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(K_e2e):
        for d_, h_ in zip(inputs, hin):
            d_.copy_(h_, non_blocking=True)
        step()
        for d_, h_ in zip(result_t, hout):
            h_.copy_(d_, non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(f0.elapsed_time(f1), world)
    peaks, peak_kind = load_peaks()
    gbs = world * algo * K / (t_ms / 1e3) / 1e9
    c = clk.summary()
    return {
        "metric": f"{kernel} HBM throughput ({args.workload})", "value": round(gbs, 1),
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "steps_requested": args.steps,
        "ms_per_step": round(t_ms / K, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if wl["kind"] == "merge" else "bf16",
        "data": "synthetic (seeded N(0,1), drawn on device)",
        "config": {"workload": args.workload, "S": S, "H": H, "Hkv": Hkv, "D": D, "P": P,
                   "algorithmic_bytes_per_step": algo,
                   "l2": "tensors larger than L2"},
        "clocks": {"sm_mhz": c["sm_mhz"], "sm_max_mhz": c["sm_max_mhz"],
                   "reasons": c["reasons"], "samples": c["samples"]},
        "gpu_launches": K * launches,
        "e2e": {"value": round(world * algo * K_e2e / (e2e_ms / 1e3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in inputs),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in result_t),
                "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs, "link_gbs_min_max": link_spread,
                "host_numa_node": numa_node},
        "roofline": {"kernel": kernel, "bound": "hbm", "achieved": round(gbs / world, 1),
                     "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                     "frac": round(gbs / world / float(peaks["hbm_gbs"]), 4), "traffic": None,
                     "note": f"peak = hbm_gbs of {peak_kind} MEASURED_PEAKS (copy bandwidth)"},
    }


def run_reference(args, wl, rank, world):
    """The fp64 oracle as it stands on the host cores, same metric and unit."""
    if rank != 0:
        return None
    vals, secs = [], []
    cores = len(os.sched_getaffinity(0))
    desc = ""
    bwd = wl["kind"] in ("ring_bwd", "ring_train")
    qkv = None if bwd else host_inputs(wl)
    # one step = one oracle call of the same size the cpu_baseline leg times
    # (ORACLE_ROWS_PER_CALL rows), so both report the same rate
    for i in range(args.warmup + args.steps):
        if bwd:
            val, desc, cores, spent, _ = cpu_oracle_bwd_sample(
                wl, budget_s=math.inf, seed=i, with_forward=wl["kind"] == "ring_train",
                max_calls=1)
        else:
            val, desc, cores, spent, _ = cpu_oracle_sample(wl, qkv, budget_s=math.inf, seed=i,
                                                           max_calls=1)
        if i >= args.warmup:
            vals.append(val)
            secs.append(spent)
    # rate of all timed steps together: FLOPs / seconds summed over steps
    v = sum(x * t for x, t in zip(vals, secs)) / sum(secs)
    S = wl["S"]
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.fmean(secs), 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/k/v, handbook make_qkv recipe)",
        "config": {"workload": args.workload, "S": S, "H": wl["H"], "Hkv": wl["Hkv"],
                   "D": wl["D"], "P": wl["P"], "layout": wl["layout"]},
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step: {desc}; {args.steps} timed steps"},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="ring128k_zigzag", choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of CPU oracle time for the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-timed-s", type=float, default=2.0,
                    help="time at least this long (more than --steps steps for short "
                         "workloads) so that the 200 ms clock sampler covers the timed region")
    ap.add_argument("--host-groups", type=int, default=8,
                    help="head groups of the host-buffer ring in the end-to-end measurement")
    args = ap.parse_args()
    wl = WORKLOADS[args.workload]
    rank, world, local = dist_info()
    if args.warmup < 3 and args.impl == "native":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return 0
        else:
            import torch
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend)
    if args.impl == "reference":
        res = run_reference(args, wl, rank, 1)
        res["n_gpus"] = args.gpus
    else:
        runner = {"merge": run_hbm, "permute": run_hbm, "ring_bwd": run_bwd,
                  "ring_train": run_bwd}.get(wl["kind"], run_gpu)
        res = runner(args, wl, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
