"""Benchmark of the KDA forward on one GB300 (or N independent replicas).

One step = one pass of the whole prefill hot path over the one-layer K3
workload (B=1, T=8192, H=96, dk=dv=128, bf16 q/k/v/z/beta, fp32 state and h0):
  kda_chunk_fwd_gated (q, k, v, z, beta, h0 -> o, hT; the gate formed inside)
or, with --path separate, kda_gate (z -> g) then kda_chunk_fwd; the other path is
timed beside it.
Inputs are resident in HBM when the timed region starts and are larger than
L2 (z, q, k, v are 201 MB each), so no L2 flush is needed between steps.

The JSON line also carries
  * roofline -- the dominant kernel's algorithmic bytes per launch over its mean
    CUDA-event duration (timed on its launching stream), against the measured
    HBM copy bandwidth; plus the whole step against the method's byte floor;
  * decode -- the decode step (512 sequences x 96 heads, fp32 state in place),
    achieved HBM GB/s against the same peak;
  * e2e -- the same prefill metric through the public API with host buffers
    (pinned host -> device copies of the step's inputs, device -> host copy of
    o and hT inside the timed region; device buffers are double-buffered so that
    one step's upload overlaps the previous step's compute and download);
  * cpu_baseline -- the fp64 oracle on the host cores over a bounded sample, and
    (one_thread) on a single thread over two heads.

``--impl reference`` times the oracle alone (the reference arm of this build).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

D = 128
TC_UNIT_BYTES = 73728  # bf16 tiles the tensor-core prep kernel writes per (chunk, head)
METRIC = "KDA prefill tokens/s (H=96,d=128) and % roofline; decode-step HBM GB/s"


# ------------------------------------------------------------------ byte counts
def prefill_bytes_per_token_head(io_bytes: int = 2, dk: int = D, dv: int = D) -> int:
    """Algorithmic HBM bytes of kda_chunk_fwd per token and head: q, k, v and o in
    the input dtype, g in fp32, beta in the input dtype."""
    return (2 * dk + dv) * io_bytes + dk * 4 + io_bytes + dv * io_bytes


def gate_bytes_per_token_head(z_bytes: int = 2, dk: int = D) -> int:
    """Algorithmic bytes of kda_gate: z read in its dtype, g written in fp32."""
    return dk * z_bytes + dk * 4


def fused_prefill_bytes_per_token_head(io_bytes: int = 2, dk: int = D, dv: int = D) -> int:
    """Algorithmic bytes of the fused-gate prefill (kda_chunk_fwd_gated) per token
    and head: q, k, v, z, beta and o in the input dtype (g is never stored)."""
    return (3 * dk + dv) * io_bytes + io_bytes + dv * io_bytes


def state_bytes(dk: int = D, dv: int = D) -> int:
    return dk * dv * 4


def decode_bytes_per_head_step(dk: int = D, dv: int = D) -> int:
    """Decode: fp32 state read + written, q, k (bf16, dk each), v and o (bf16, dv
    each), g (fp32, dk), beta (bf16)."""
    return 2 * state_bytes(dk, dv) + 2 * dk * 2 + 2 * dv * 2 + dk * 4 + 2


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------------- clocks
class _Nvml:
    """Read-only NVML queries through ctypes (SM clock, its maximum, and the active
    clock-event reasons): fast enough to sample short timed regions.  Nothing is
    ever set."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}

    def __init__(self, index: int):
        import ctypes
        self.ok = False
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if self.lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) != 0:
                return
            self.ct = ctypes
            self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except (OSError, AttributeError):
            pass

    def sample(self):
        ct = self.ct
        sm, mx, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(sm)) != 0:  # NVML_CLOCK_SM
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, ct.byref(mx))
        self.reasons_fn(self.handle, ct.byref(rs))
        return float(sm.value), float(mx.value), int(rs.value)


class ClockSampler:
    """Samples SM clocks and clock-event reasons while timed regions are open:
    NVML every 5 ms when libnvidia-ml is loadable, else nvidia-smi every 200 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int = 0):
        self.gpu = gpu_index
        self.samples = []  # (time, sm MHz, max MHz, set of reasons)
        self._stop = threading.Event()
        self._thr = None
        self.marks = []
        self.source = None

    def start(self):
        self._thr = threading.Thread(target=self._run, daemon=True)
        self._thr.start()

    def mark(self, on: bool):
        self.marks.append((time.time(), on))

    def _run(self):
        nv = _Nvml(self.gpu)
        self.source = "nvml" if nv.ok else "nvidia-smi"
        while not self._stop.is_set():
            try:
                if nv.ok:
                    r = nv.sample()
                    if r:
                        reasons = {n for bit, n in _Nvml.REASONS.items() if r[2] & bit}
                        self.samples.append((time.time(), r[0], r[1], reasons))
                    self._stop.wait(0.005)
                    continue
                out = subprocess.run(["nvidia-smi", "-i", str(self.gpu),
                                      f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits"],
                                     capture_output=True, text=True, timeout=5).stdout.strip()
                if out:
                    f = [x.strip() for x in out.split(",")]
                    reasons = {n for i, n in enumerate(self.NAMES)
                               if len(f) > 5 + i and f[5 + i].lower().startswith("active")}
                    if _isnum(f[1]) and _isnum(f[2]):
                        self.samples.append((time.time(), float(f[1]), float(f[2]), reasons))
            except Exception:
                pass
            self._stop.wait(0.2)

    def stop(self):
        self._stop.set()
        if self._thr:
            self._thr.join(timeout=10)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clocks unavailable"]}
        # samples taken while a timed region was open
        spans, t_on = [], None
        for t, on in self.marks:
            if on:
                t_on = t
            elif t_on is not None:
                spans.append((t_on, t))
                t_on = None
        inside = [x for x in self.samples if any(a <= x[0] <= b for a, b in spans)]
        use = inside or self.samples
        reasons = set().union(*[x[3] for x in use])
        return {"sm_mhz": statistics.median([x[1] for x in use]),
                "sm_max_mhz": max(x[2] for x in use), "reasons": sorted(reasons),
                "samples": len(inside), "source": self.source}


def _isnum(x):
    try:
        float(x)
        return True
    except ValueError:
        return False


# ------------------------------------------------------------- measured traffic
def kernel_traffic(name: str):
    """Per-launch DRAM bytes of `name` from the committed ncu summary, if the
    summary's source hash still matches the kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(rf"^\|\s*{re.escape(name)}\s*\|\s*([0-9.eE+]+)\s*\|\s*([0-9a-f]+)\s*\|", text,
                  re.M)
    if not m:
        return None
    src = os.path.join(ROOT, "chunked_gated_delta_fwd_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(src)):
        if f.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(src, f), "rb").read())
    if h.hexdigest()[:12] != m.group(2):
        return None
    return float(m.group(1))


# ------------------------------------------------------------------------ arms
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The maximum of x over all ranks of the default process group (x itself on
    one rank): the job's time is that of its slowest rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args):
    """The oracle, timed on the host cores over a bounded sample of the workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import torch

    import oracle
    import workloads

    w = workloads.prefill()
    heads = args.ref_heads
    T = w.seq_lens[0]
    gen = torch.Generator().manual_seed(w.seed)
    # same distributions as the GPU workload, drawn for the sampled heads only
    q = torch.nn.functional.normalize(torch.randn(T, heads, D, generator=gen), dim=-1).bfloat16()
    k = torch.nn.functional.normalize(torch.randn(T, heads, D, generator=gen), dim=-1).bfloat16()
    v = torch.randn(T, heads, D, generator=gen).bfloat16()
    z = torch.randn(T, heads, D, generator=gen).bfloat16()
    beta = torch.sigmoid(torch.randn(T, heads, generator=gen)).bfloat16()
    A = torch.rand(heads, generator=gen) * 2 - 1
    h0 = torch.randn(1, heads, D, D, generator=gen) * 0.02
    cores = os.cpu_count() or 1
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        g = oracle.gate(z, A)
        oracle.recurrence(q, k, v, g, beta, h0, n_threads=cores)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    per_step = statistics.median(times)
    tokens_per_s = T * heads / per_step / w.H  # H=96 tokens/s equivalent
    line = {
        "impl": "reference", "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        # measured: one step is the sample below (heads of the 96), median over steps
        "ms_per_step": per_step * 1e3,
        # the same time scaled to all 96 heads (the time a whole step would take)
        "ms_per_step_scaled_to_all_heads": per_step * 1e3 * w.H / heads,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": f"{heads} of {w.H} heads x {T} tokens",
                   "global_batch": 1, "seq_len": T, "parallelism": "none (host cores)"},
        "cpu_baseline": {"value": tokens_per_s, "unit": "tokens/s", "cores": min(cores, heads),
                         "kind": "oracle",
                         "sample": f"gate + fp64 recurrence over {heads} heads x {T} tokens, "
                                   f"scaled to H={w.H}"},
        "e2e": {"value": tokens_per_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def cpu_baseline(heads=96, T=8192, seed=1002):
    """fp64 oracle over a bounded sample (heads x T tokens), scaled to H=96."""
    import torch

    import oracle

    gen = torch.Generator().manual_seed(seed)
    q = torch.nn.functional.normalize(torch.randn(T, heads, D, generator=gen), dim=-1).bfloat16()
    k = torch.nn.functional.normalize(torch.randn(T, heads, D, generator=gen), dim=-1).bfloat16()
    v = torch.randn(T, heads, D, generator=gen).bfloat16()
    z = torch.randn(T, heads, D, generator=gen).bfloat16()
    beta = torch.sigmoid(torch.randn(T, heads, generator=gen)).bfloat16()
    A = torch.rand(heads, generator=gen) * 2 - 1
    cores = os.cpu_count() or 1
    t0 = time.perf_counter()
    g = oracle.gate(z, A)
    oracle.recurrence(q, k, v, g, beta, None, n_threads=cores)
    dt = time.perf_counter() - t0
    # the same oracle on one thread, over the first two heads
    t1 = time.perf_counter()
    oracle.recurrence(q[:, :2], k[:, :2], v[:, :2], g[:, :2], beta[:, :2], None, n_threads=1)
    dt1 = time.perf_counter() - t1
    return {"value": T * heads / dt / 96, "unit": "tokens/s", "cores": min(cores, heads),
            "kind": "oracle",
            "sample": f"gate + fp64 recurrence, {heads} heads x {T} tokens "
                      f"({dt:.1f} s), scaled to H=96",
            "one_thread": {"value": T * 2 / dt1 / 96, "unit": "tokens/s",
                           "sample": f"fp64 recurrence, 2 heads x {T} tokens ({dt1:.2f} s), "
                                     f"scaled to H=96"}}


def run_gpu(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import chunked_gated_delta_fwd_gb300 as kda
    import workloads

    hbm_peak, bf16_peak, peak_src = load_peaks()
    w = workloads.prefill()
    inp = workloads.make_inputs(w, dev)
    NT, H = w.n_tokens, w.H
    ws = torch.empty(kda.chunk_fwd_workspace_size(NT, 1, H, torch.bfloat16), dtype=torch.uint8,
                     device=dev)
    g = torch.empty(NT, H, D, dtype=torch.float32, device=dev)
    o = torch.empty(NT, H, D, dtype=torch.bfloat16, device=dev)
    hT = torch.empty(1, H, D, D, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step_separate():
        kda.gate(inp["z"], inp["A"], out=g)
        kda.chunk_fwd(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"], inp["cu_seqlens"],
                      workspace=ws, out=o, final_state_out=hT)

    def step_fused():
        kda.chunk_fwd_gated(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"], inp["beta"],
                            inp["h0"], inp["cu_seqlens"], workspace=ws, out=o,
                            final_state_out=hT)

    fused = args.path == "fused"
    step, alt_step = (step_fused, step_separate) if fused else (step_separate, step_fused)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    def timed(fn, steps, warmup):
        for _ in range(warmup):
            fn()
        barrier()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        clocks.mark(True)
        start.record(stream)
        for _ in range(steps):
            fn()
        stop.record(stream)
        barrier()
        clocks.mark(False)
        return max_over_ranks(start.elapsed_time(stop) / steps, world, dev)

    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    ms_step = timed(step, args.steps, args.warmup)
    tokens_per_s = NT * world / (ms_step * 1e-3)
    ms_alt = timed(alt_step, args.steps, args.warmup)

    # per-kernel event timing pass (same steps, profiling on)
    kda.profile_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    per_kernel = kda.profile_collect()
    kda.profile_enable(False)
    launches = sum(n for n, _ in per_kernel.values())
    dom_name, (dom_n, dom_ms) = max(per_kernel.items(), key=lambda kv: kv[1][1])
    dom_avg_ms = dom_ms / dom_n
    tok_heads = NT * H
    units = (NT // 64) * H  # (chunk, head) units of this single-sequence workload
    # The method's algorithmic bytes for one step (the inputs read once, o and hT
    # written once, h0 read once; no workspace intermediates): 1,282 B per
    # token-head with the gate fused (z in bf16), 1,538 B with g read in fp32 (plus
    # the gate kernel's own z read and g write on the separate path).
    if fused:
        step_bytes = tok_heads * fused_prefill_bytes_per_token_head(2) + 2 * H * state_bytes()
    else:
        step_bytes = tok_heads * (prefill_bytes_per_token_head(2)
                                  + gate_bytes_per_token_head(2)) + 2 * H * state_bytes()
    step_floor_ms = step_bytes / (hbm_peak * 1e9) * 1e3
    # Each kernel's own input/output bytes, workspace tiles included (what a
    # kernel on its own would have to move; context for the measured traffic).
    tile_bytes = units * (TC_UNIT_BYTES + D * 4)
    kernel_io_bytes = {
        "kda_gate": tok_heads * gate_bytes_per_token_head(2),
        "kda_tc_prep": tok_heads * (prefill_bytes_per_token_head(2) - D * 2) + tile_bytes,
        "kda_tc_prep_gated": tok_heads * (fused_prefill_bytes_per_token_head(2) - D * 2)
        + tile_bytes,
        "kda_tc_chain": tile_bytes + tok_heads * D * 2 + 2 * H * state_bytes(),
    }
    # The roofline line follows the method's byte count: the step's algorithmic
    # bytes over the dominant kernel's mean launch time (one launch per step).
    alg_bytes = step_bytes
    achieved = alg_bytes / (dom_avg_ms * 1e-3) / 1e9

    # decode step (512 x 96, fp32 state, in place)
    dw = workloads.decode()
    S = workloads.make_decode_state(dw, dev)
    dinp = workloads.make_decode_step(dw, 0, dev)
    dg = kda.gate(dinp["z"], dinp["A"])
    do = torch.empty(dw.N, dw.H, D, dtype=torch.bfloat16, device=dev)

    def dstep():
        kda.recurrent_step(dinp["q"], dinp["k"], dinp["v"], dg, dinp["beta"], S, out=do)

    # 100 in-place steps, each on fresh seeded inputs (made beforehand, ~75 MB a step),
    # each timed on its own with events; the median step is reported
    n_dec = 100
    dsteps = [workloads.make_decode_step(dw, i, dev) for i in range(n_dec)]
    dgs = [kda.gate(x["z"], x["A"]) for x in dsteps]
    for _ in range(args.warmup):
        dstep()
    barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_dec)]
    clocks.mark(True)
    for (e0, e1), x, gx in zip(evs, dsteps, dgs):
        e0.record(stream)
        kda.recurrent_step(x["q"], x["k"], x["v"], gx, x["beta"], S, out=do)
        e1.record(stream)
    barrier()
    clocks.mark(False)
    dec_times = [e0.elapsed_time(e1) for e0, e1 in evs]
    ms_dec = max_over_ranks(statistics.median(dec_times), world, dev)
    ms_dec_mean = max_over_ranks(sum(dec_times) / n_dec, world, dev)
    del dsteps, dgs
    dec_bytes = dw.N * dw.H * decode_bytes_per_head_step()
    dec_gbs = dec_bytes / (ms_dec * 1e-3) / 1e9

    # four tokens per sequence in one pass over the state (speculative verify + commit)
    TM = 4
    mq = {k_: v_.unsqueeze(1).expand(dw.N, TM, *v_.shape[1:]).contiguous()
          for k_, v_ in dinp.items() if k_ in ("q", "k", "v", "beta")}
    mg = dg.unsqueeze(1).expand(dw.N, TM, *dg.shape[1:]).contiguous()
    mo = torch.empty(dw.N, TM, dw.H, D, dtype=torch.bfloat16, device=dev)

    def mstep():
        kda.recurrent_multi_step(mq["q"], mq["k"], mq["v"], mg, mq["beta"], S, out=mo)

    ms_multi = timed(mstep, max(args.steps, 20), args.warmup)
    multi_bytes = dw.N * dw.H * (2 * state_bytes() + TM * (decode_bytes_per_head_step()
                                                           - 2 * state_bytes()))
    multi_gbs = multi_bytes / (ms_multi * 1e-3) / 1e9
    del S

    # the method's other prefill workloads: one timed fused prefill each, inputs in HBM
    # (reported beside the headline, not part of it)
    other = {}
    if not args.skip_other_workloads:
        # the headline prefill (gate already applied) with and without the state
        # written every 512 tokens (prefix-cache checkpoints)
        kda.gate(inp["z"], inp["A"], out=g)
        ck = torch.empty(NT // 512, H, D, D, dtype=torch.float32, device=dev)

        def step_plain():
            kda.chunk_fwd(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                          inp["cu_seqlens"], workspace=ws, out=o, final_state_out=hT)

        def step_ckpt():
            kda.chunk_fwd_checkpointed(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                                       inp["cu_seqlens"], ckpt_tokens=512,
                                       ckpt_capacity=NT // 512, ckpt_out=ck, workspace=ws,
                                       out=o, final_state_out=hT)

        ms_plain = timed(step_plain, args.steps, args.warmup)
        ms_ck = timed(step_ckpt, args.steps, args.warmup)
        other["prefill_checkpoints_512"] = {
            "checkpoints": NT // 512, "checkpoint_bytes": ck.numel() * 4,
            "ms_per_step": ms_ck, "ms_per_step_without": ms_plain}
        del ck
        # the same prefill with q, k normalised in the kernel and the output
        # RMSNorm x Sigmoid gate applied before the store (gate logits read in bf16)
        gz = torch.randn(NT, H, D, device=dev).to(torch.bfloat16)
        nw = torch.ones(D, device=dev)

        def step_all_fused():
            kda.chunk_fwd_fused(inp["q"], inp["k"], inp["v"], inp["beta"], inp["h0"],
                                inp["cu_seqlens"], z=inp["z"], A=inp["A"], qk_l2_eps=1e-6,
                                out_gate=gz, out_norm_weight=nw, out_norm_eps=1e-6,
                                workspace=ws, out=o, final_state_out=hT)

        ms_fz = timed(step_all_fused, args.steps, args.warmup)

        # the headline step with the precise state update (KDA_CHUNK_PRECISE: Kt in
        # fp32, tf32 state-update MMAs); its own, larger workspace
        ws_p = torch.empty(kda.chunk_fwd_workspace_size(NT, 1, H, torch.bfloat16, kda.PRECISE),
                           dtype=torch.uint8, device=dev)

        def step_precise():
            kda.chunk_fwd_fused(inp["q"], inp["k"], inp["v"], inp["beta"], inp["h0"],
                                inp["cu_seqlens"], z=inp["z"], A=inp["A"], workspace=ws_p,
                                out=o, final_state_out=hT, flags=kda.PRECISE)

        ms_pr = timed(step_precise, args.steps, args.warmup)
        other["prefill_precise_state"] = {
            "ms_per_step": ms_pr, "ms_per_step_default": ms_step if fused else ms_alt,
            "workspace_bytes": ws_p.numel(), "workspace_bytes_default": ws.numel()}
        del ws_p
        other["prefill_qk_norm_output_gate"] = {
            "ms_per_step": ms_fz, "ms_per_step_gated_only": ms_step if fused else ms_alt,
            "extra_bytes_per_token_head": D * 2,
            "step_floor_ms": (NT * H * (fused_prefill_bytes_per_token_head(2) + D * 2)
                              + 2 * H * state_bytes()) / (hbm_peak * 1e9) * 1e3}
        del gz

        for wl in (workloads.varlen(), workloads.long_context()):
            inp2 = workloads.make_inputs(wl, dev)
            N2 = wl.n_seqs
            ws2 = torch.empty(kda.chunk_fwd_workspace_size(wl.n_tokens, N2, wl.H, torch.bfloat16),
                              dtype=torch.uint8, device=dev)
            o2 = torch.empty(wl.n_tokens, wl.H, D, dtype=torch.bfloat16, device=dev)
            hT2 = torch.empty(N2, wl.H, D, D, dtype=torch.float32, device=dev)

            def step2():
                kda.chunk_fwd_gated(inp2["q"], inp2["k"], inp2["v"], inp2["z"], inp2["A"],
                                    inp2["beta"], inp2["h0"], inp2["cu_seqlens"], workspace=ws2,
                                    out=o2, final_state_out=hT2)

            ms2 = timed(step2, 3, 3)
            tok_heads2 = wl.n_tokens * wl.H
            floor2 = (tok_heads2 * fused_prefill_bytes_per_token_head(2)
                      + (2 if inp2["h0"] is not None else 1) * N2 * wl.H * state_bytes()) \
                / (hbm_peak * 1e9) * 1e3
            other[wl.name] = {"tokens": wl.n_tokens, "sequences": N2, "heads": wl.H,
                              "ms_per_step": ms2, "tokens_per_s": wl.n_tokens * world / (ms2 * 1e-3),
                              "step_floor_ms": floor2, "step_frac": floor2 / ms2}
            del inp2, ws2, o2, hT2
            torch.cuda.empty_cache()

    # end to end through the public API with host buffers
    pin = {k: v.cpu().pin_memory() for k, v in inp.items() if isinstance(v, torch.Tensor)
           and k in ("z", "q", "k", "v", "beta", "A", "h0", "cu_seqlens")}
    o_host = torch.empty(NT, H, D, dtype=torch.bfloat16).pin_memory()
    hT_host = torch.empty(1, H, D, D, dtype=torch.float32).pin_memory()
    # two sets of device inputs and outputs: step i uses set i % 2, so the upload of
    # step i + 1 runs while step i computes and downloads (each step still copies
    # its own inputs in and its own results out inside the timed region; the
    # compute stream is idle when the region opens, so no copy precedes its start)
    dsets = [{k: torch.empty_like(v, device=dev) for k, v in pin.items()} for _ in range(2)]
    osets = [(torch.empty(NT, H, D, dtype=torch.bfloat16, device=dev),
              torch.empty(1, H, D, D, dtype=torch.float32, device=dev)) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d2h = o_host.numel() * 2 + hT_host.numel() * 4

    # the large inputs are copied in slices on four copy streams (several copies in
    # flight); the results go back on their own stream
    copy_streams = [torch.cuda.Stream(dev) for _ in range(4)]
    d2h_stream = torch.cuda.Stream(dev)

    def slices_of(dbuf):
        out = []
        for k_, v_ in pin.items():
            n_sl = 4 if v_.numel() * v_.element_size() > (64 << 20) else 1
            for part in torch.tensor_split(torch.arange(v_.shape[0]), n_sl):
                if part.numel():
                    a_, b_ = int(part[0]), int(part[-1]) + 1
                    out.append((dbuf[k_][a_:b_], v_[a_:b_]))
        return out

    slice_sets = [slices_of(d_) for d_ in dsets]
    freed = [None, None]  # per set: the compute that last read it
    n_e2e = [0]

    def e2e_step():
        i = n_e2e[0]
        n_e2e[0] += 1
        sid = i % 2
        dbuf, (o_d, hT_d) = dsets[sid], osets[sid]
        # upload: may start once the step that last used this set has computed
        done = []
        for j, (dst, src) in enumerate(slice_sets[sid]):
            cs = copy_streams[j % len(copy_streams)]
            if freed[sid] is not None:
                cs.wait_event(freed[sid])
            with torch.cuda.stream(cs):
                dst.copy_(src, non_blocking=True)
        for cs in copy_streams:
            ev = torch.cuda.Event()
            ev.record(cs)
            done.append(ev)
        for ev in done:
            stream.wait_event(ev)
        if fused:
            kda.chunk_fwd_gated(dbuf["q"], dbuf["k"], dbuf["v"], dbuf["z"], dbuf["A"],
                                dbuf["beta"], dbuf["h0"], dbuf["cu_seqlens"], workspace=ws,
                                out=o_d, final_state_out=hT_d)
        else:
            kda.gate(dbuf["z"], dbuf["A"], out=g)
            kda.chunk_fwd(dbuf["q"], dbuf["k"], dbuf["v"], g, dbuf["beta"], dbuf["h0"],
                          dbuf["cu_seqlens"], workspace=ws, out=o_d, final_state_out=hT_d)
        computed = torch.cuda.Event()
        computed.record(stream)
        freed[sid] = computed
        # download this step's results; the next step's compute (and the end of the
        # timed region) waits for it
        d2h_stream.wait_event(computed)
        with torch.cuda.stream(d2h_stream):
            o_host.copy_(o_d, non_blocking=True)
            hT_host.copy_(hT_d, non_blocking=True)
        fetched = torch.cuda.Event()
        fetched.record(d2h_stream)
        stream.wait_event(fetched)

    ms_e2e = timed(e2e_step, max(3, args.steps // 4), max(3, args.warmup))
    clocks.stop()
    e2e_tps = NT * world / (ms_e2e * 1e-3)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline()
    traffic = kernel_traffic(dom_name)
    # measured DRAM bytes of one step: the captured kernels (the plan kernel moves a
    # few KB and is not captured), per launch x launches per step
    step_traffic = None
    big = [k_ for k_ in per_kernel if k_ != "kda_plan"]
    parts = [kernel_traffic(k_) for k_ in big]
    if parts and all(p_ is not None for p_ in parts):
        step_traffic = sum(p_ * per_kernel[k_][0] / args.steps for p_, k_ in zip(parts, big))
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "global_batch": world, "seq_len": NT, "heads": H,
                   "dk": D, "dv": D, "chunk": 64,
                   "step": "kda_chunk_fwd_gated (gate fused)" if fused
                   else "kda_gate + kda_chunk_fwd",
                   "l2": "inputs larger than L2 (201 MB per q/k/v/z tensor), no flush",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": dom_name, "achieved": achieved,
                     "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
                     "traffic": traffic,
                     "traffic_over_alg": (traffic / alg_bytes) if traffic else None,
                     "alg_bytes_per_launch": alg_bytes,
                     "alg_bytes_rule": ("step bytes of the method per launch: "
                                        + ("1282" if fused else "1538 + 768 (gate)")
                                        + " B per token-head x token-heads + h0 and hT"),
                     "kernel_io_bytes": kernel_io_bytes.get(dom_name),
                     "mean_launch_ms": dom_avg_ms,
                     "peak_source": f"{peak_src} hbm_gbs (copy, burst)",
                     "step_floor_ms": step_floor_ms, "step_frac": step_floor_ms / ms_step,
                     "step_traffic": step_traffic,
                     "step_traffic_over_alg": (step_traffic / step_bytes) if step_traffic
                     else None},
        "kernels": {k: {"launches": n, "mean_ms": t / n} for k, (n, t) in per_kernel.items()},
        "alt_step": {"step": "kda_gate + kda_chunk_fwd" if fused
                     else "kda_chunk_fwd_gated (gate fused)", "ms_per_step": ms_alt,
                     "value": NT * world / (ms_alt * 1e-3)},
        "other_workloads": other,
        "decode": {"workload": dw.name, "ms_per_step": ms_dec, "achieved_gbs": dec_gbs,
                   "peak_gbs": hbm_peak, "frac": dec_gbs / hbm_peak,
                   "bytes_per_step": dec_bytes, "steps": n_dec, "mean_ms": ms_dec_mean,
                   "timing": "median of 100 in-place steps, each on fresh seeded inputs",
                   "multi_token": {"tokens_per_sequence": TM, "ms_per_step": ms_multi,
                                   "achieved_gbs": multi_gbs, "frac": multi_gbs / hbm_peak,
                                   "ms_per_token": ms_multi / TM}},
        "e2e": {"value": e2e_tps, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e},
        "gpu_launches": launches,
        "cpu_baseline": cpu,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_profile_case(args):
    """A small case for ncu captures (a few GB on the device at most, inputs above
    L2): one decode step on N=128 x H=96 (0.8 GB state), then --reps prefill steps
    (fused gate, and gate + chunk) on B=1, T=8192, H=32 bf16.  Prints one line."""
    import torch

    import chunked_gated_delta_fwd_gb300 as kda
    import workloads

    dev = torch.device("cuda", 0)
    dw = workloads.DecodeWorkload("profile decode", N=128, H=96)
    S = workloads.make_decode_state(dw, dev)
    di = workloads.make_decode_step(dw, 0, dev)
    dg = kda.gate(di["z"], di["A"])
    kda.recurrent_step(di["q"], di["k"], di["v"], dg, di["beta"], S)
    torch.cuda.synchronize(dev)
    del S
    w = workloads.custom([8192], H=32, dtype=torch.bfloat16, seed=3, h0_std=0.02)
    inp = workloads.make_inputs(w, dev)
    gz = torch.randn(w.n_tokens, w.H, D, device=dev).to(torch.bfloat16)
    for _ in range(args.reps):
        o, hT = kda.chunk_fwd_gated(inp["q"], inp["k"], inp["v"], inp["z"], inp["A"],
                                    inp["beta"], inp["h0"], inp["cu_seqlens"])
        g = kda.gate(inp["z"], inp["A"])
        o2, _ = kda.chunk_fwd(inp["q"], inp["k"], inp["v"], g, inp["beta"], inp["h0"],
                              inp["cu_seqlens"])
        # the output gate applied by the chain, and the precise state update
        kda.chunk_fwd_fused(inp["q"], inp["k"], inp["v"], inp["beta"], inp["h0"],
                            inp["cu_seqlens"], z=inp["z"], A=inp["A"], out_gate=gz)
        kda.chunk_fwd_fused(inp["q"], inp["k"], inp["v"], inp["beta"], inp["h0"],
                            inp["cu_seqlens"], z=inp["z"], A=inp["A"], flags=kda.PRECISE)
    torch.cuda.synchronize(dev)
    kda.get_device_error()
    print(json.dumps({"profile_case": "decode N=128 H=96; prefill B=1 T=8192 H=32 "
                      "(gate fused; gate + chunk; output gate in the chain; precise)",
                      "reps": args.reps, "o_mean_abs": float(o.float().abs().mean()),
                      "paths_max_diff": float((o.float() - o2.float()).abs().max())}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--ref-heads", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", choices=["fused", "separate"], default="fused",
                    help="prefill step: gate fused into the chunk kernels, or kda_gate then "
                         "kda_chunk_fwd (the other one is timed too, as alt_step)")
    ap.add_argument("--skip-other-workloads", action="store_true",
                    help="do not time the varlen and long-context prefills beside the headline")
    ap.add_argument("--profile-case", action="store_true",
                    help="run the small profiling case (for ncu captures) instead of the bench")
    ap.add_argument("--reps", type=int, default=2, help="prefill steps of --profile-case")
    args = ap.parse_args(argv)
    if args.profile_case:
        return run_profile_case(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
