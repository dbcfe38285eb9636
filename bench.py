"""Benchmark of the packed variable-length gated-delta layer on GB300.

One step = one gdn_layer_varlen call (conv -> prepare -> recurrence) over one
batch of the workload, inputs resident in HBM.  Default workload: the decode
step (64 sequences x 1 token, HQ=16, H=32, K=V=128, bf16, fp32 state
[64,32,128,128] carried in place).  Prints ONE JSON line (rank 0).  With the
default workload the line also carries, under "workloads", the same
measurement of the prefill (8 x 4096), ragged (32 x U[1, 8192]) and long
(1 x 131072, V=256, D=2) workloads, whose dominant kernel is the chunked
tensor-core kernel (roofline against the bf16 tensor peak).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the fp64 CPU oracle, timed on host cores)

Multi-GPU: one process per GPU (torchrun); every rank runs its own batch of
the workload (independent sequences: no data-path collective), so scaling is
weak; value = tokens of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "prefill", "ragged", "long", "tiny"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="the default (decode) line without the prefill, ragged and long "
                         "records")
    ap.add_argument("--rule", default="gated_delta",
                    choices=["gated_delta", "delta", "gated", "linear"],
                    help="update rule (delta: no decay; gated: no retrieval; linear: neither)")
    ap.add_argument("--gate", default="scalar", choices=["scalar", "per_channel"],
                    help="per_channel: the layer with one decay logit per key channel, "
                         "a [N, H, K] (GDN_OPT_GATE_PER_CHANNEL)")
    ap.add_argument("--dense", default=None, choices=["scalar", "per_channel"],
                    help="time the dense-layout call (q, k, v [B, S, H, n]) on the workload's "
                         "batch and head geometry (equal lengths), scalar or per-channel gate")
    ap.add_argument("--capture", type=int, default=0,
                    help="state-update capture capacity (1..8): time gdn_layer_varlen_capture "
                         "with every sequence asking for that many tokens")
    ap.add_argument("--chunk-min-len", type=int, default=None,
                    help="sequences of at least this many tokens take a chunked kernel "
                         "(gdn_set_chunk_min_len; a large value keeps every sequence "
                         "token-serial)")
    ap.add_argument("--lens", default=None,
                    help="comma-separated sequence lengths replacing the workload's "
                         "(same head geometry and distributions; for small profiling cases)")
    return ap.parse_args()


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _replica_seed(wl, rank):
    """Each rank's replica draws its own batch (weak scaling, no shared work)."""
    return wl.seed + 1000 * rank


def _max_over_ranks(values, device):
    """Per-rank timings -> their maximum over the ranks of the process group
    (unchanged without one); the job is as slow as its slowest replica."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def _job_tokens_per_s(world, tokens_per_rank, steps, ms):
    """Whole-job throughput: the tokens of all ranks over the max-over-ranks time."""
    return world * tokens_per_rank * steps / (ms * 1e-3)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def capture_bytes(wl, B, cap):
    """Bytes a capture of capacity cap adds to the token-serial kernel: the
    capsule and the conv capture rows written in full, the captured raw rows read."""
    if cap <= 0:
        return 0
    esz = 2 if wl.dtype == "bf16" else 4
    capsule = B * cap * (wl.H + wl.HQ * wl.K + wl.H * wl.V) * 4
    rows = B * cap * wl.width * esz
    return capsule + 2 * rows


def algorithmic_bytes_delta(wl, N, B, cap=0, per_channel=False):
    """Bytes the token-serial recurrence kernel must move per launch in the
    layer call (it also writes the final conv state and any capture; with the
    per-channel gate it reads the decay logits a [N, H, K])."""
    esz = 2 if wl.dtype == "bf16" else 4
    state = 2 * B * wl.H * wl.V * wl.K * 4            # read + write fp32 state
    qk = N * wl.HQ * 2 * wl.K * 4                     # normalised q and k (fp32)
    gb = N * wl.H * 2 * 4                             # g and beta
    v = N * wl.H * wl.V * esz                         # v columns of the conv output
    out = N * wl.H * wl.V * esz
    conv_state = 2 * B * wl.width * wl.L * esz        # final conv state: read + write
    pc = N * wl.H * wl.K * 4 if per_channel else 0
    return state + qk + gb + v + out + conv_state + pc + capture_bytes(wl, B, cap)


def algorithmic_bytes_delta_pc(wl, N, B):
    """Bytes the per-channel chunked recurrence (prepare + scan kernels) must
    move per launch pair: the conv output's q, k and v columns, the decay
    logits a [N, H, K] and beta logits, the output and the fp32 state in and
    out.  The chunk images the prepare kernel writes and the scan kernel reads
    back are the design's own traffic, not counted."""
    esz = 2 if wl.dtype == "bf16" else 4
    state = 2 * B * wl.H * wl.V * wl.K * 4
    qkv = N * (2 * wl.HQ * wl.K + wl.H * wl.V) * esz
    logits = N * wl.H * (wl.K + 1) * 4
    out = N * wl.H * wl.V * esz
    return state + qkv + logits + out


def algorithmic_bytes_layer(wl, N, B):
    """Bytes the whole layer must move per step (inputs read once, outputs written once)."""
    esz = 2 if wl.dtype == "bf16" else 4
    W = wl.width
    return (N * W * esz                               # qkv
            + W * wl.Kc * esz + W * esz               # conv weight, bias
            + 2 * B * W * wl.L * esz                  # conv state in / out
            + 2 * N * wl.H * 4 + 2 * wl.H * 4         # a, b, A_log, dt_bias
            + 2 * B * wl.H * wl.V * wl.K * 4          # delta state in / out
            + N * wl.H * wl.V * esz)                  # out


def chunked_flops(wl, N):
    """Contraction FLOPs of the chunked form counted at the canonical chunk
    C = 64 (whatever chunk the kernel uses): per token and value head
    2C(3K + 2V) (K K^T, T K', Q K^T; T V', P U) + 6KV (W S^T, Q S^T, U^T K')."""
    C = 64
    return N * wl.H * (2 * C * (3 * wl.K + 2 * wl.V) + 6 * wl.K * wl.V)


def _profile_traffic(kernel, workload):
    """Per-launch DRAM bytes from the committed ncu summary, if it still
    describes the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    info = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                info[k.strip()] = v.strip()
    src = info.get("source_file")
    sha = info.get("source_sha256")
    tb = info.get("traffic_bytes_per_launch")
    if not (src and sha and tb):
        return None
    with open(os.path.join(ROOT, src), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != sha:
            return None
    return int(float(tb))


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"gdn_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = max(mx, float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def run_reference(args, wl):
    """The fp64 CPU oracle, timed as it stands on this host's cores."""
    import numpy as np
    import torch

    import oracle
    from varlen_gated_delta_gb300 import workloads as W

    world, rank, _ = _dist()
    if rank != 0:
        return
    sample_wl, sample = _oracle_sample(wl)
    d = W.make_inputs(sample_wl, "cpu")
    c = lambda t: None if t is None else t.double().numpy()
    inputs = [c(d[k]) for k in ("qkv", "w", "bias", "a", "b", "A_log", "dt_bias")]
    offs = np.asarray(d["offsets_list"], np.int32)
    ci, si = c(d["conv_init"]), c(d["state_init"])
    act = "bf16" if sample_wl.dtype == "bf16" else "f32"

    cap = args.capture
    counts = np.full(len(offs) - 1, cap, np.int32)
    opts = {"gated_delta": 0, "delta": 1, "gated": 2, "linear": 3}[args.rule]

    def step():
        if opts:
            oracle.layer_varlen_ex(*inputs, offs, ci, si, sample_wl.H, sample_wl.HQ, sample_wl.K,
                                   sample_wl.V, sample_wl.Kc, sample_wl.D, opts,
                                   silu=sample_wl.silu, scale=d["scale"], act_dtype=act)
        elif cap:
            oracle.layer_varlen_capture(*inputs, offs, ci, si, sample_wl.H, sample_wl.HQ,
                                        sample_wl.K, sample_wl.V, sample_wl.Kc, sample_wl.D,
                                        counts, cap, silu=sample_wl.silu, scale=d["scale"],
                                        act_dtype=act)
        else:
            oracle.layer_varlen(*inputs, offs, ci, si, sample_wl.H, sample_wl.HQ, sample_wl.K,
                                sample_wl.V, sample_wl.Kc, sample_wl.D, silu=sample_wl.silu,
                                scale=d["scale"], act_dtype=act)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    toks = sample_wl.N * args.steps
    value = toks / dt
    line = {
        "impl": "reference", "metric": "gated-delta layer tokens/s", "value": value,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "sample": sample, **({"capture": cap} if cap else {}),
                   **({"rule": args.rule} if opts else {})},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _oracle_sample(wl):
    """A bounded slice of the workload for the CPU oracle (about a second a step)."""
    from varlen_gated_delta_gb300 import workloads as W
    if wl.name == "decode":
        return wl, "the whole decode batch (64 sequences x 1 token, all 32 heads)"
    if wl.name == "tiny":
        return wl, "the whole tiny batch"
    # prefill-like workloads: one 256-token sequence with the workload's head geometry
    s = W.scaled(wl, (256,), name=wl.name + "-sample")
    return s, f"one 256-token sequence of the {wl.name} geometry (HQ={wl.HQ}, H={wl.H}, K={wl.K}, V={wl.V})"


def cpu_baseline(wl, budget_s=12.0):
    """The fp64 oracle, as it stands, on a bounded sample of the workload
    (``_oracle_sample``), repeated for about ``budget_s`` seconds."""
    import numpy as np

    import oracle
    from varlen_gated_delta_gb300 import workloads as W
    sample_wl, sample = _oracle_sample(wl)
    d = W.make_inputs(sample_wl, "cpu")
    c = lambda t: None if t is None else t.double().numpy()
    inputs = [c(d[k]) for k in ("qkv", "w", "bias", "a", "b", "A_log", "dt_bias")]
    offs = np.asarray(d["offsets_list"], np.int32)
    ci, si = c(d["conv_init"]), c(d["state_init"])
    act = "bf16" if sample_wl.dtype == "bf16" else "f32"
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.layer_varlen(*inputs, offs, ci, si, sample_wl.H, sample_wl.HQ, sample_wl.K,
                            sample_wl.V, sample_wl.Kc, sample_wl.D, silu=sample_wl.silu,
                            scale=d["scale"], act_dtype=act)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or reps >= 200:
            break
    return {"value": sample_wl.N * reps / dt, "unit": "tokens/s", "cores": oracle.threads(),
            "kind": "oracle", "sample": f"{sample}; {reps} repetitions in {dt:.1f} s"}


def _measure(args, wl, dev, world, rank, local, gdn, W):
    """One workload through gdn_layer_varlen: device-resident steps (CUDA graph
    replays), the dominant kernel alone (library events inside the same
    replays) and the end-to-end run with host buffers.  Returns the record of
    rank 0 (None elsewhere).

    The layer carries its states in place, as a decode loop does.  Two
    independent state sets alternate from step to step, so the state a step
    reads was last touched two steps earlier, with at least one full state
    (268 MB on the decode batch, more than the 129 MB L2) streamed in between:
    no step finds the state it reads still in L2."""
    import torch
    import torch.distributed as dist

    d = W.make_inputs(wl, dev, seed=_replica_seed(wl, rank))
    offs = d["offsets_list"]
    N, B = offs[-1], len(offs) - 1
    act = gdn.GDN_ACT_SILU if wl.silu else gdn.GDN_ACT_NONE
    out = torch.empty((N, wl.H, wl.V), dtype=wl.torch_dtype, device=dev)
    conv_states = [d["conv_init"], d["conv_init"].clone()]
    states = [d["state_init"], d["state_init"].clone()]
    cap = args.capture
    if cap:
        counts = torch.full((B,), cap, dtype=torch.int32, device=dev)
        conv_upd = torch.empty((B, cap, wl.width), dtype=wl.torch_dtype, device=dev)
        capsule = torch.empty((B, cap * (wl.H + wl.HQ * wl.K + wl.H * wl.V)),
                              dtype=torch.float32, device=dev)

    opts = gdn.RULE_OPTS[args.rule]
    if args.gate == "per_channel":  # one decay logit per key channel
        opts |= gdn.GDN_OPT_GATE_PER_CHANNEL
        gpc = torch.Generator(device=dev).manual_seed(wl.seed + 500)
        d["a"] = torch.randn((N, wl.H, wl.K), generator=gpc, device=dev) * wl.a_std + wl.a_mean
    # (with the per-channel gate the workspace also holds the chunk images of
    # its chunked form)
    ws = torch.empty(gdn.gdn_workspace_bytes_ex(B, N, wl.H, wl.HQ, wl.K, wl.V, wl.Kc, wl.D,
                                                gdn.GDN_BF16 if wl.dtype == "bf16" else gdn.GDN_F32,
                                                opts),
                     dtype=torch.uint8, device=dev)

    def call(qkv, a, b, offsets, sset, out_t=None, capsule_t=None):
        # decode-style carry: the final states overwrite the initial ones in place
        out_t = out if out_t is None else out_t
        conv_state, state = conv_states[sset], states[sset]
        kw = dict(H=wl.H, HQ=wl.HQ, K=wl.K, V=wl.V, Kc=wl.Kc, D=wl.D, act=act,
                  scale=d["scale"], offsets_host=offs, out=out_t, conv_fin=conv_state,
                  state_fin=state, workspace=ws)
        if opts:
            gdn.gdn_layer_varlen_ex(qkv, d["w"], d["bias"], a, b, d["A_log"], d["dt_bias"],
                                    offsets, conv_state, state, opts=opts, cap=cap,
                                    counts=counts if cap else None,
                                    conv_updates=conv_upd if cap else None,
                                    capsule=(capsule if capsule_t is None else capsule_t)
                                    if cap else None, **kw)
        elif cap:
            gdn.gdn_layer_varlen_capture(qkv, d["w"], d["bias"], a, b, d["A_log"], d["dt_bias"],
                                         offsets, conv_state, state, counts, cap=cap,
                                         conv_updates=conv_upd,
                                         capsule=capsule if capsule_t is None else capsule_t, **kw)
        else:
            gdn.gdn_layer_varlen(qkv, d["w"], d["bias"], a, b, d["A_log"], d["dt_bias"],
                                 offsets, conv_state, state, **kw)

    def step(sset):
        call(d["qkv"], d["a"], d["b"], d["offsets"], sset)

    stream = torch.cuda.current_stream(dev)
    warm = max(3, args.warmup)
    for i in range(warm):
        step(i & 1)
    torch.cuda.synchronize()
    gdn.gdn_workspace_status(ws)

    # eager steps (one library call per step from Python)
    eager0, eager1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    eager0.record(stream)
    for i in range(args.steps):
        step(i & 1)
    eager1.record(stream)
    torch.cuda.synchronize()
    eager_ms = eager0.elapsed_time(eager1)

    # each state set's step captured once in a CUDA graph (launch-bound
    # decode), replayed alternately
    launches_per_step0 = gdn.gdn_launch_count()
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step(0)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    launches_per_step = gdn.gdn_launch_count() - launches_per_step0
    graphs = []
    for sset in (0, 1):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(sset)
        graphs.append(g)
    for i in range(warm):
        graphs[i & 1].replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        graphs[i & 1].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = launches_per_step * args.steps
    ms = e0.elapsed_time(e1)

    # dominant kernel, timed inside the same layer calls with CUDA events the
    # library records on its stream right around that kernel's launch; the
    # other state set's step runs between two timed steps, as in the timed run
    dom = (gdn.GDN_KERNEL_SERIAL if max(wl.lengths()) < gdn.gdn_chunk_min_len()
           else gdn.GDN_KERNEL_CHUNKED)
    k_start = torch.cuda.Event(enable_timing=True)
    k_stop = torch.cuda.Event(enable_timing=True)
    k_start.record(stream)
    k_stop.record(stream)
    torch.cuda.synchronize()
    kern_ms = []
    gdn.gdn_set_kernel_events(dom, k_start, k_stop)
    try:
        # captured in a graph like the timed steps, so no CPU gap sits inside
        kgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(kgraph):
            step(0)
    finally:
        gdn.gdn_set_kernel_events(dom, None, None)
    for i in range(warm + args.steps):
        graphs[1].replay()
        kgraph.replay()
        if i >= warm:
            torch.cuda.synchronize()
            kern_ms.append(k_start.elapsed_time(k_stop))
    clocks = sampler.stop()

    # end to end through the public API with host buffers: every step copies its
    # inputs in from pinned host memory and reads its output (and capsule) back.
    # The copies run on two copy streams into double-buffered device buffers, so
    # that step i+1's inputs arrive and step i-1's output leaves while step i
    # computes (the serving pattern); events order each buffer's reuse.
    host = {k: d[k].cpu().pin_memory() for k in ("qkv", "a", "b")}
    host_offs = d["offsets"].cpu().pin_memory()
    dev_in = [{k: torch.empty_like(d[k]) for k in ("qkv", "a", "b")} for _ in range(2)]
    dev_offs = [torch.empty_like(d["offsets"]) for _ in range(2)]
    outs = [out, torch.empty_like(out)]
    out_host = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + host_offs.numel() * 4
    d2h = out_host[0].numel() * out_host[0].element_size()
    if cap:  # the caller also reads the capsule back
        caps = [capsule, torch.empty_like(capsule)]
        capsule_host = [torch.empty(capsule.shape, dtype=capsule.dtype, pin_memory=True)
                        for _ in range(2)]
        d2h += capsule_host[0].numel() * 4
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: [torch.cuda.Event() for _ in range(2)]
    in_ready, in_free, out_ready, out_free = ev(), ev(), ev(), ev()

    def e2e_step(i, comp):
        j = i & 1
        with torch.cuda.stream(h2d_s):
            if i >= 2:  # buffer j was last read by step i - 2 of this run
                h2d_s.wait_event(in_free[j])
                # step i - 2's output has left too: the compute stream then joins
                # one other stream per step (this copy), off its critical path
                h2d_s.wait_event(out_free[j])
            for k in host:
                dev_in[j][k].copy_(host[k], non_blocking=True)
            dev_offs[j].copy_(host_offs, non_blocking=True)
            in_ready[j].record(h2d_s)
        comp.wait_event(in_ready[j])
        call(dev_in[j]["qkv"], dev_in[j]["a"], dev_in[j]["b"], dev_offs[j], j, out_t=outs[j],
             capsule_t=caps[j] if cap else None)
        in_free[j].record(comp)
        out_ready[j].record(comp)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(out_ready[j])
            out_host[j].copy_(outs[j], non_blocking=True)
            if cap:
                capsule_host[j].copy_(caps[j], non_blocking=True)
            out_free[j].record(d2h_s)

    def e2e_run(steps):
        comp = torch.cuda.current_stream(dev)
        h2d_s.wait_stream(comp)
        d2h_s.wait_stream(comp)
        for i in range(steps):
            e2e_step(i, comp)
        comp.wait_stream(h2d_s)
        comp.wait_stream(d2h_s)

    e2e_run(3)
    torch.cuda.synchronize()
    # Small steps (decode) are bound by launch and cross-stream latency: there
    # the whole pipelined run (every step's copies in, call and read-back) is
    # captured once as a CUDA graph, whose copy nodes move the pinned host
    # buffers on every replay.
    small = h2d + d2h < (4 << 20)
    if small:
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph):
            e2e_run(args.steps)
        e2e_graph.replay()
        torch.cuda.synchronize()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    if small:
        e2e_graph.replay()
    else:
        e2e_run(args.steps)
    x1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = x0.elapsed_time(x1)
    last = (args.steps - 1) & 1
    # the last step's output and capsule, read back on the host, are this step's results
    torch.testing.assert_close(out_host[last].to(dev), outs[last], rtol=0, atol=0)

    ms, e2e_ms = _max_over_ranks([ms, e2e_ms], dev)
    if rank != 0:
        return None
    hbm, tf, tf_s, peak_src = _peaks()
    kavg = statistics.mean(kern_ms)
    value = _job_tokens_per_s(world, N, args.steps, ms)
    if dom == gdn.GDN_KERNEL_SERIAL:
        kbytes = algorithmic_bytes_delta(wl, N, B, cap, per_channel=args.gate == "per_channel")
        achieved = kbytes / (kavg * 1e-3) / 1e9
        roof = {"kernel": "delta_serial_kernel", "bound": "hbm", "achieved": achieved,
                "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": None if cap else _profile_traffic("delta_serial", wl.name),
                "algorithmic_bytes": kbytes, "kernel_ms": kavg,
                "peak_source": f"hbm_gbs of {peak_src}"}
    elif args.gate == "per_channel":
        kbytes = algorithmic_bytes_delta_pc(wl, N, B)
        achieved = kbytes / (kavg * 1e-3) / 1e9
        roof = {"kernel": "pc_prep_kernel + pc_scan_kernel", "bound": "hbm", "achieved": achieved,
                "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
                "algorithmic_bytes": kbytes, "kernel_ms": kavg,
                "peak_source": f"hbm_gbs of {peak_src}"}
    else:
        kflops = chunked_flops(wl, N)
        achieved = kflops / (kavg * 1e-3) / 1e12
        roof = {"kernel": "chunked_delta_kernel", "bound": "tensor", "achieved": achieved,
                "peak": tf, "unit": "TFLOP/s", "frac": achieved / tf,
                "traffic": _profile_traffic("chunked_delta", wl.name),
                "algorithmic_flops": kflops, "kernel_ms": kavg,
                "peak_source": f"bf16_tflops (burst) of {peak_src}"}
    rec = {
        "metric": "gated-delta layer tokens/s", "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": warm,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "B": B, "N": N, "HQ": wl.HQ, "H": wl.H, "K": wl.K,
                   "V": wl.V, "Kc": wl.Kc, "D": wl.D,
                   "state_carry": "in place, two state sets alternating",
                   "l2": "inputs larger than L2 (129 MB); the state a step reads was last "
                         "touched two steps before",
                   "parallelism": f"replicas x{world}",
                   **({"capture": cap} if cap else {}),
                   **({"rule": args.rule} if args.rule != "gated_delta" else {}),
                   **({"gate": "per_channel"} if args.gate == "per_channel" else {}),
                   **({"chunk_min_len": args.chunk_min_len}
                      if args.chunk_min_len is not None else {})},
        "layer_gbs": algorithmic_bytes_layer(wl, N, B) / (ms * 1e-3 / args.steps) / 1e9,
        "roofline": roof,
        "e2e": {"value": _job_tokens_per_s(world, N, args.steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipeline": "copies on two streams, double-buffered, overlapping the "
                            "neighbouring steps' compute" +
                            (" (the whole run replayed as one CUDA graph)" if small else "")},
        "gpu_launches": launches,
        "timing": "CUDA graph replay of one gdn_layer_varlen%s call per step"
                  % ("_ex" if opts else "_capture" if cap else ""),
        "ms_per_step_eager": eager_ms / args.steps,
        "clocks": clocks,
    }
    return rec


# Workloads measured beside the default (decode) one in the same JSON line,
# so that one run reports both halves of the metric: decode (HBM-bound) and
# prefill (tensor-core bound).
EXTRA_WORKLOADS = ("prefill", "ragged", "long")


def run_ours(args, wl):
    import torch
    import torch.distributed as dist

    import varlen_gated_delta_gb300 as gdn
    from varlen_gated_delta_gb300 import build as gdn_build
    from varlen_gated_delta_gb300 import workloads as W

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0:
        gdn_build.build()
    if world > 1:
        dist.barrier()
    gdn.load_library()
    if args.chunk_min_len is not None:
        gdn.gdn_set_chunk_min_len(args.chunk_min_len)

    line = _measure(args, wl, dev, world, rank, local, gdn, W)
    extras = {}
    plain = not (args.lens or args.capture or args.rule != "gated_delta"
                 or args.gate != "scalar" or args.chunk_min_len is not None)
    if plain and wl.name == "decode" and not args.no_extra:
        for name in EXTRA_WORKLOADS:
            torch.cuda.empty_cache()
            rec = _measure(args, W.WORKLOADS[name], dev, world, rank, local, gdn, W)
            if rank == 0:
                if not args.no_cpu_baseline:
                    rec["cpu_baseline"] = cpu_baseline(W.WORKLOADS[name], budget_s=8.0)
                for k in ("n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                          "vs_baseline", "data", "metric", "unit"):
                    rec.pop(k, None)
                extras[name] = rec
        # the prefill batch with one decay logit per key channel (the
        # per-channel chunked route: prepare and scan kernels)
        pc_args = argparse.Namespace(**vars(args))
        pc_args.gate = "per_channel"
        torch.cuda.empty_cache()
        rec = _measure(pc_args, W.WORKLOADS["prefill"], dev, world, rank, local, gdn, W)
        if rank == 0:
            for k in ("n_gpus", "steps", "warmup", "higher_is_better", "scaling",
                      "vs_baseline", "data", "metric", "unit"):
                rec.pop(k, None)
            extras["prefill_per_channel"] = rec
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(wl)
        if extras:
            line["workloads"] = extras
            line["gpu_launches_all_workloads"] = line["gpu_launches"] + sum(
                r["gpu_launches"] for r in extras.values())
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_dense(args, wl):
    """The dense-layout call (rlx-cpu GatedDeltaNet thunk layout) on the
    workload's batch, length and head geometry (n = K = V, H heads for q/k/v).
    A one-GPU measurement: under torchrun only rank 0 runs it."""
    import torch

    if _dist()[1] != 0:
        return

    import varlen_gated_delta_gb300 as gdn
    from varlen_gated_delta_gb300 import build as gdn_build

    lens = wl.lengths()
    if len(set(lens)) != 1 or wl.K != wl.V:
        raise SystemExit("--dense needs equal sequence lengths and K == V")
    B, S, H, n = len(lens), lens[0], wl.H, wl.K
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gdn_build.build()
    gdn.load_library()
    g = torch.Generator(device=dev)
    g.manual_seed(wl.seed + 77)
    r = lambda *sh: torch.randn(*sh, generator=g, device=dev)
    T = wl.torch_dtype
    q, v = r(B, S, H, n).to(T), r(B, S, H, n).to(T)
    k = torch.nn.functional.normalize(r(B, S, H, n), dim=-1).to(T)
    perch = args.dense == "per_channel"
    gate = torch.sigmoid(r(B, S, H, n) + 2.0) if perch else torch.sigmoid(r(B, S, H) + 2.0)
    beta = torch.sigmoid(r(B, S, H))
    state = r(B, H, n, n) * 0.05
    out = torch.empty((B, S, H, n), dtype=T, device=dev)
    # long bf16 sequences take a chunked route through the workspace entry
    # point: packing kernel + chunked kernel (scalar gate), or packing +
    # prepare + scan kernels (per-channel gate, workspace with chunk images)
    ws_bytes = (gdn.gdn_dense_workspace_bytes_ex(B, S, H, n, gdn.GDN_BF16, perch)
                if T == torch.bfloat16 else 0)
    chunked = ws_bytes > 0 and S >= gdn.gdn_chunk_min_len()
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if chunked else None

    def step():
        gdn.gdn_gated_delta_dense(q, k, v, gate, beta, state, gate_per_channel=perch, out=out,
                                  workspace=ws)

    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        step()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    kern_ms = None
    if chunked:  # the chunked kernel alone, bracketed by events inside a replayed graph
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream)
        k1.record(stream)
        torch.cuda.synchronize()
        gdn.gdn_set_kernel_events(gdn.GDN_KERNEL_CHUNKED, k0, k1)
        try:
            kg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(kg):
                step()
        finally:
            gdn.gdn_set_kernel_events(gdn.GDN_KERNEL_CHUNKED, None, None)
        ks = []
        for i in range(max(3, args.warmup) + args.steps):
            kg.replay()
            if i >= max(3, args.warmup):
                torch.cuda.synchronize()
                ks.append(k0.elapsed_time(k1))
        kern_ms = statistics.mean(ks)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    esz = 2 if T == torch.bfloat16 else 4
    N = B * S
    kbytes = (2 * B * H * n * n * 4 + 4 * N * H * n * esz + N * H * 4
              + (N * H * n * 4 if perch else N * H * 4))
    hbm, tf, _, peak_src = _peaks()
    achieved = kbytes / (ms * 1e-3) / 1e9
    roof = {"kernel": "delta_dense_kernel", "bound": "hbm", "achieved": achieved,
            "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "traffic": None,
            "algorithmic_bytes": kbytes, "kernel_ms": ms,
            "peak_source": f"hbm_gbs of {peak_src}"}
    if chunked and perch:  # prepare + scan against the bytes they must move
        kb = (2 * B * H * n * n * 4 + 4 * N * H * n * esz + N * H * 4 + N * H * n * 4)
        ach = kb / (kern_ms * 1e-3) / 1e9
        roof = {"kernel": "pc_prep_kernel + pc_scan_kernel", "bound": "hbm", "achieved": ach,
                "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "traffic": None,
                "algorithmic_bytes": kb, "kernel_ms": kern_ms,
                "peak_source": f"hbm_gbs of {peak_src}"}
    elif chunked:
        kflops = N * H * (2 * 64 * (3 * n + 2 * n) + 6 * n * n)
        ach = kflops / (kern_ms * 1e-3) / 1e12
        roof = {"kernel": "chunked_delta_kernel", "bound": "tensor", "achieved": ach, "peak": tf,
                "unit": "TFLOP/s", "frac": ach / tf, "traffic": None, "algorithmic_flops": kflops,
                "kernel_ms": kern_ms, "peak_source": f"bf16_tflops (burst) of {peak_src}"}
    line = {
        "metric": "gated-delta dense tokens/s", "value": N / (ms * 1e-3), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic",
        "config": {"workload": f"{wl.name}-dense", "B": B, "S": S, "H": H, "n": n,
                   "gate": args.dense, "state_carry": "in place"},
        "roofline": roof,
        "route": ("packing + per-channel prepare + scan kernels" if chunked and perch else
                  "packing kernel + chunked kernel" if chunked else "token-serial dense kernel"),
        "timing": "CUDA graph replay of one gdn_gated_delta_dense%s call per step"
                  % ("_ws" if chunked else ""),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def main():
    args = _args()
    from varlen_gated_delta_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    if args.lens:
        wl = W.scaled(wl, [int(x) for x in args.lens.split(",")],
                      name=f"{wl.name}-{args.lens.replace(',', 'x')}")
    if args.impl == "reference":
        run_reference(args, wl)
    elif args.dense:
        run_dense(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
