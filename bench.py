"""Throughput of the attention hot path on GB300 (one JSON line on rank 0).

A step is one pass over every kernel of the path on synthetic inputs resident
in HBM:
  * prefill - Llama-3-8B-shaped causal GQA prefill, B=4 S=8192 n_h=32 n_kv=8
    D_h=128 bf16, RoPE base 5e5 (attn_prefill: the RoPE pass writing rotated
    keys, then the tensor-core attention kernel);
  * gqa     - GQA decode, 59 sequences with 4096..8192 cached keys, n_h=32
    n_kv=8 D_h=128 bf16 (attn_decode: split-KV partials + combine);
  * mla     - MLA-absorbed decode, 32 sequences x 32768 keys, 128 heads over
    one 576-dim latent head, V = its first 512 dims (attn_decode);
  * gpt2    - GPT-2-small-shaped causal MHA prefill, B=8 S=1024 n_h=n_kv=12
    D_h=64 bf16, no RoPE (attn_prefill).
``value`` is the Llama prefill throughput in TFLOP/s (causal FLOPs = half the
dense 4*B*n_h*S^2*D_h); the decode calls report KV GB/s (algorithmic cache
bytes) and the GPT-2 prefill TFLOP/s in ``parts``.  Every input of the first
three parts is larger than the 129 MB L2; the GPT-2 part's 48 MB is not, so an
L2 flush (a 256 MB write, outside its events) precedes each of its calls.

``cpu_baseline`` times the fp64 oracle on the host cores on every one of the
five configurations: the tiny and GPT-2 prefills in full, the Llama prefill on
sampled blocks of query rows, the decodes on a subset of their sequences.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--extras]

--extras prints a different line instead: the calls outside the step (chunked,
windowed, split-halves-RoPE, MLA and GPT-2-shaped prefill, windowed decode, the
RoPE pass, the fused KV append, and whole decode steps that append the new
token before attending), each against its roofline on one GPU.

--impl reference times the fp64 CPU oracle on the host cores instead (each
step: a block of 256 query rows of one (batch, head) slice of the prefill
workload, all their visible keys).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "prefill causal-attn TFLOP/s and decode KV GB/s on 1 GB300, % of roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}

# DRAM bytes (read + write) per launch of the prefill kernel on the benchmark
# workload, from an ncu capture of one launch; valid only for the kernel source
# it was taken on (sha256 of prefill_tc.cu, first 16 hex digits), else null.
PREFILL_TRAFFIC = {"kernel_sha": "68782a22c8d249d6", "bytes": 1.8346e9 + 232.63e6}


def kernel_sha(name: str) -> str:
    path = os.path.join(ROOT, "transformer_causal_attention_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    return FALLBACK_PEAKS, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ distributed
def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle (CPU) baseline
def oracle_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_prefill_rows(q, k, v, cfg, b, h, rows):
    """The oracle on a block of query rows of one (batch, head) slice of the
    prefill workload; returns (seconds, causal FLOPs of those rows: 4*D_h per
    visible key, i.e. 2*D_h for q.k and 2*D_h for the weighted value)."""
    import oracle
    t0 = time.perf_counter()
    oracle.attention_prefill_rows(q, k, v, b, h, rows, rope_base=cfg["rope_base"], scale=cfg["scale"])
    dt = time.perf_counter() - t0
    return dt, float(sum(4.0 * cfg["D_h"] * (m + 1) for m in rows))


def sample_rows(cfg, i, n_rows=256):
    """The i-th sample: n_rows consecutive query rows of (b, h), spread over the sequence."""
    b, h = i % cfg["B"], (7 * i) % cfg["n_h"]
    n_blocks = cfg["S"] // n_rows
    r0 = ((5 * i + 3) % n_blocks) * n_rows
    return b, h, list(range(r0, r0 + n_rows))


def cpu_baseline_prefill(q, k, v, cfg, budget_s: float = 8.0, max_samples: int = 512):
    done, secs, flops = 0, 0.0, 0.0
    while done < max_samples and (done == 0 or secs < budget_s):
        b, h, rows = sample_rows(cfg, done)
        dt, fl = oracle_prefill_rows(q, k, v, cfg, b, h, rows)
        secs += dt
        flops += fl
        done += 1
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{done} blocks of 256 query rows from different (batch, head) slices of the prefill "
                      f"workload (all visible keys each), fp64, {secs:.1f} s"}


def cpu_baseline_decode(q, kc, vc, sl, cfg, n_seq: int):
    import oracle
    idx = list(range(n_seq))
    t0 = time.perf_counter()
    oracle.attention_decode(q, kc, vc, sl.numpy(), rope_base=cfg["rope_base"], rope_offset=cfg["rope_offset"],
                            rope_dims=cfg["rope_dims"], scale=cfg["scale"], batch_index=idx)
    dt = time.perf_counter() - t0
    by = workloads.decode_bytes(cfg, sl[:n_seq].tolist())
    return {"value": by / dt / 1e9, "unit": "GB/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"{n_seq} of {cfg['B']} sequences, fp64, {dt:.1f} s"}


def cpu_baseline_full_prefill(cfg, min_s: float = 0.5):
    """The oracle on a whole prefill configuration, repeated until min_s has passed."""
    import oracle
    q, k, v = workloads.prefill_inputs(cfg, seed=0)
    runs, secs = 0, 0.0
    while runs == 0 or secs < min_s:
        t0 = time.perf_counter()
        oracle.attention_prefill(q, k, v, rope_base=cfg["rope_base"], scale=cfg["scale"])
        secs += time.perf_counter() - t0
        runs += 1
    flops = runs * workloads.causal_flops(cfg["B"], cfg["S"], cfg["n_h"], cfg["D_h"])
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"the whole configuration, {runs} run(s), fp64 from {cfg['dtype']} inputs, {secs:.2f} s"}


# ------------------------------------------------------------------ reference arm
# The workload both arms report (the reference arm times the oracle on samples of its prefill).
WORKLOAD = ("llama3-8b-shaped causal GQA prefill B=4 S=8192 n_h=32 n_kv=8 D_h=128 RoPE 5e5"
            " + GQA decode 59 seqs L~U[4096,8192] n_h=32 n_kv=8 D_h=128"
            " + MLA-absorbed decode 32 seqs x 32768 keys, 128 heads, 576/512 latent"
            " + GPT-2-small-shaped causal MHA prefill B=8 S=1024 n_h=12 D_h=64")


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cfg = workloads.config("llama3_8b")
    q, k, v = workloads.prefill_inputs(cfg, seed=0)
    for i in range(args.warmup):
        b, h, rows = sample_rows(cfg, i)
        oracle_prefill_rows(q, k, v, cfg, b, h, rows)
    secs, flops = 0.0, 0.0
    for i in range(args.steps):
        b, h, rows = sample_rows(cfg, args.warmup + i)
        dt, fl = oracle_prefill_rows(q, k, v, cfg, b, h, rows)
        secs += dt
        flops += fl
    value = flops / secs / 1e12
    sample = "each step: 256 consecutive query rows of one (batch, head) slice of the prefill workload, fp64"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "l2": "n/a (host cores)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm
def run_ours(args):
    import torch
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import transformer_causal_attention_gb300 as attn
    lib = attn.load()

    peaks, peak_kind = load_peaks()
    stream = torch.cuda.current_stream()

    # ---- inputs (seeded, CPU-drawn, then resident in HBM)
    pc = workloads.config("llama3_8b", B=args.prefill_batch)
    q_h, k_h, v_h = workloads.prefill_inputs(pc, seed=rank)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    out = torch.empty_like(q)
    k_rot = torch.empty_like(k)
    gc = workloads.config("gqa_decode")
    if "gqa" not in args.parts:
        gc = workloads.config("gqa_decode", B=1, max_len=256, len_lo=1, len_hi=256)
    gq_h, gkc_h, gvc_h, gsl_h = workloads.decode_inputs(gc, seed=rank)
    gq, gkc, gvc, gsl = gq_h.to(dev), gkc_h.to(dev), gvc_h.to(dev), gsl_h.to(dev)
    gout = torch.empty(gc["B"], gc["n_h"], gc["D_v"], dtype=torch.bfloat16, device=dev)
    gws = torch.empty(attn.decode_workspace_size(gc["B"], gc["n_h"], gc["n_kv"], gc["D_qk"], gc["D_v"],
                                                 gc["max_len"]), dtype=torch.uint8, device=dev)
    mc = workloads.config("mla_decode")
    if "mla" not in args.parts:
        mc = workloads.config("mla_decode", B=1, max_len=256, len_lo=1, len_hi=256)
    mq_h, mkc_h, _, msl_h = workloads.decode_inputs(mc, seed=rank)
    mq, mkc, msl = mq_h.to(dev), mkc_h.to(dev), msl_h.to(dev)
    mvc = mkc[..., :mc["D_v"]]
    mout = torch.empty(mc["B"], mc["n_h"], mc["D_v"], dtype=torch.bfloat16, device=dev)
    mws = torch.empty(attn.decode_workspace_size(mc["B"], mc["n_h"], mc["n_kv"], mc["D_qk"], mc["D_v"],
                                                 mc["max_len"]), dtype=torch.uint8, device=dev)

    g2 = workloads.config("gpt2")
    g2q_h, g2k_h, g2v_h = workloads.prefill_inputs(g2, seed=rank)
    g2q, g2k, g2v = g2q_h.to(dev), g2k_h.to(dev), g2v_h.to(dev)
    g2out = torch.empty_like(g2q)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # > L2: the GPT-2 inputs are 48 MB

    def prefill():
        attn.prefill(q, k, v, rope_base=pc["rope_base"], scale=pc["scale"], out=out, k_rot=k_rot, stream=stream)

    def gpt2():
        attn.prefill(g2q, g2k, g2v, scale=g2["scale"], out=g2out, stream=stream)

    def gqa():
        attn.decode(gq, gkc, gvc, gsl, rope_base=gc["rope_base"], rope_offset=0, rope_dims=gc["rope_dims"],
                    scale=gc["scale"], out=gout, workspace=gws, stream=stream)

    def mla():
        attn.decode(mq, mkc, mvc, msl, rope_base=mc["rope_base"], rope_offset=mc["rope_offset"],
                    rope_dims=mc["rope_dims"], scale=mc["scale"], out=mout, workspace=mws, stream=stream)

    parts = [(n, fn) for n, fn in (("prefill", prefill), ("gqa", gqa), ("mla", mla), ("gpt2", gpt2))
             if n in args.parts]
    for _ in range(args.warmup):
        for name, fn in parts:
            if name == "gpt2":
                flush.zero_()  # as in the timed steps: its first launch loads the fill kernel's module
            fn()
    torch.cuda.synchronize()

    # ---- timed region: K steps, events around every call on the launching stream
    ev = {name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)] for name, _ in parts}
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    launches0 = attn.launch_count()
    barrier(world)
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        for name, fn in parts:
            if name == "gpt2":
                flush.zero_()  # its inputs fit in L2: evict them, outside its events
            a, b = ev[name][i]
            a.record(stream)
            fn()
            b.record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = attn.launch_count() - launches0
    clocks = sampler.stop()
    if attn.device_status() != 0:
        raise RuntimeError("a kernel reported a device-side wait timeout")

    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    part_ms = {name: max_over_ranks(sum(a.elapsed_time(b) for a, b in ev[name]), world) / args.steps
               for name, _ in parts}
    for name in ("prefill", "gqa", "mla", "gpt2"):
        part_ms.setdefault(name, float("nan"))
    pf_flops = workloads.causal_flops(pc["B"], pc["S"], pc["n_h"], pc["D_h"])
    g_bytes = workloads.decode_bytes(gc, gsl_h.tolist())
    m_bytes = workloads.decode_bytes(mc, msl_h.tolist())
    prefill_tflops = world * pf_flops / (part_ms["prefill"] * 1e-3) / 1e12
    gqa_gbs = world * g_bytes / (part_ms["gqa"] * 1e-3) / 1e9
    mla_gbs = world * m_bytes / (part_ms["mla"] * 1e-3) / 1e9
    mla_tflops = world * workloads.decode_flops(mc, msl_h.tolist()) / (part_ms["mla"] * 1e-3) / 1e12
    gpt2_tflops = world * workloads.causal_flops(g2["B"], g2["S"], g2["n_h"], g2["D_h"]) / (part_ms["gpt2"] * 1e-3) / 1e12

    hbm_peak = float(peaks["hbm_gbs"])
    bf16_peak = float(peaks["bf16_tflops"])
    traffic = PREFILL_TRAFFIC["bytes"] if PREFILL_TRAFFIC["kernel_sha"] == kernel_sha("prefill_tc.cu") else None
    per_gpu_prefill = prefill_tflops / world
    roofline = {"bound": "tensor", "achieved": per_gpu_prefill, "peak": bf16_peak, "unit": "TFLOP/s",
                "frac": per_gpu_prefill / bf16_peak, "traffic": traffic,
                "kernel": "attn_prefill (RoPE-K pass + prefill_tc_kernel<128>)",
                "peak_source": f"{peak_kind} bf16 burst"}

    # ---- end to end through the public API: pinned host inputs in, result out, every step.
    # The batch is pipelined per sequence over three streams: the copy-in of
    # sequence i+1 and the copy-out of sequence i-1 overlap the prefill of i, and
    # consecutive steps overlap too: a sequence's copy-in waits only for the previous
    # step's prefill of that sequence (which read its device buffers), and its prefill
    # only for the previous step's copy-out of its output.
    e2e = None
    if not args.no_e2e and "prefill" in args.parts:
        qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
        outp = torch.empty(q_h.shape, dtype=q_h.dtype).pin_memory()
        e2e_steps = max(3, min(args.steps, 10))
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        nb = pc["B"]
        prev_done, prev_copied = [None] * nb, [None] * nb

        def e2e_step():
            loaded = [torch.cuda.Event() for _ in range(nb)]
            done = [torch.cuda.Event() for _ in range(nb)]
            copied = [torch.cuda.Event() for _ in range(nb)]
            for b in range(nb):
                if prev_done[b] is not None:
                    s_in.wait_event(prev_done[b])  # the previous step's prefill of b read these buffers
                with torch.cuda.stream(s_in):
                    q[b].copy_(qp[b], non_blocking=True)
                    k[b].copy_(kp[b], non_blocking=True)
                    v[b].copy_(vp[b], non_blocking=True)
                    loaded[b].record(s_in)
            for b in range(nb):
                stream.wait_event(loaded[b])
                if prev_copied[b] is not None:
                    stream.wait_event(prev_copied[b])  # the previous step's output of b has been read
                attn.prefill(q[b:b + 1], k[b:b + 1], v[b:b + 1], rope_base=pc["rope_base"], scale=pc["scale"],
                             out=out[b:b + 1], k_rot=k_rot[b:b + 1], stream=stream)
                done[b].record(stream)
            for b in range(nb):
                s_out.wait_event(done[b])
                with torch.cuda.stream(s_out):
                    outp[b].copy_(out[b], non_blocking=True)
                    copied[b].record(s_out)
            prev_done[:] = done
            prev_copied[:] = copied

        e2e_step()
        torch.cuda.synchronize()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for _ in range(e2e_steps):
            e2e_step()
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)  # the last step's outputs are in host memory
        b_.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b_), world) / e2e_steps
        h2d = sum(t.numel() * t.element_size() for t in (qp, kp, vp))
        e2e = {"value": world * pf_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": outp.numel() * outp.element_size(),
               "ms_per_step": e2e_ms,
               "method": "pinned host Q/K/V copied in and the output copied out every step, pipelined per "
                         "sequence over three streams (copy-in, prefill, copy-out), consecutive steps "
                         "overlapping where their buffers allow"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_prefill(q_h, k_h, v_h, pc)
        cpu["configs"] = {
            "tiny": cpu_baseline_full_prefill(workloads.config("tiny")),
            "gpt2": cpu_baseline_full_prefill(g2, min_s=0.0),
            "llama3_8b": {key: cpu[key] for key in ("value", "unit", "cores", "kind", "sample")},
            "gqa_decode": cpu_baseline_decode(gq_h, gkc_h, gvc_h, gsl_h, gc, n_seq=min(16, gc["B"])),
            "mla_decode": cpu_baseline_decode(mq_h, mkc_h, mkc_h[..., :mc["D_v"]], msl_h, mc, n_seq=min(8, mc["B"])),
        }

    if rank == 0:
        line = {
            "metric": METRIC, "value": prefill_tflops, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD,
                       "l2": "prefill, GQA and MLA decode inputs larger than L2 (129 MB), no flush; "
                             "the GPT-2 part: a 256 MB flush write before each call, outside its events",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "parts": {
                "prefill": {"ms": part_ms["prefill"], "value": prefill_tflops, "unit": "TFLOP/s",
                            "frac_of_peak": per_gpu_prefill / bf16_peak},
                "gqa_decode": {"ms": part_ms["gqa"], "value": gqa_gbs, "unit": "GB/s",
                               "roofline": {"bound": "hbm", "achieved": gqa_gbs / world, "peak": hbm_peak,
                                            "unit": "GB/s", "frac": gqa_gbs / world / hbm_peak}},
                "mla_decode": {"ms": part_ms["mla"], "value": mla_gbs, "unit": "GB/s", "tflops": mla_tflops,
                               "roofline": {"bound": "hbm", "achieved": mla_gbs / world, "peak": hbm_peak,
                                            "unit": "GB/s", "frac": mla_gbs / world / hbm_peak}},
                "gpt2": {"ms": part_ms["gpt2"], "value": gpt2_tflops, "unit": "TFLOP/s",
                         "roofline": {"bound": "tensor", "achieved": gpt2_tflops / world, "peak": bf16_peak,
                                      "unit": "TFLOP/s", "frac": gpt2_tflops / world / bf16_peak},
                         "l2": "256 MB flush write before each call, outside its events"},
            },
            "roofline": roofline,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "gpu_launches": int(launches),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ extra rows (opt-in)
def visible_pairs(q_pos, n_keys, window=None, n_sink=0):
    """(query, key) pairs a causal mask admits for queries at positions q_pos over
    keys 0..n_keys-1; with a window, key n is visible from m when n <= m and
    (m - n < window or n < n_sink)."""
    total = 0
    for m in q_pos:
        hi = min(m, n_keys - 1) + 1
        if window is None:
            total += hi
        else:
            in_win = min(hi, window)
            total += in_win + min(n_sink, max(0, hi - window))
    return float(total)


def window_decode_keys(L: int, window: int, n_sink: int) -> int:
    """Keys a decode query at position L - 1 sees: L - 1 - n < window, or n < n_sink."""
    return min(L, window) + min(n_sink, max(0, L - window))


def run_extras(args):
    """One JSON line timing the calls outside the default step, each on its own
    workload against its roofline.  L2 is flushed (a 256 MB write) before every
    timed call, outside the events."""
    import torch
    if int(os.environ.get("RANK", "0")) != 0:  # one GPU's figures; under torchrun rank 0 alone runs
        return 0
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import transformer_causal_attention_gb300 as attn
    attn.load()
    peaks, peak_kind = load_peaks()
    hbm_peak, bf16_peak = float(peaks["hbm_gbs"]), float(peaks["bf16_tflops"])
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        total = 0.0
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            total += a.elapsed_time(b)
        if attn.device_status() != 0:
            raise RuntimeError("a kernel reported a device-side wait timeout")
        return total / args.steps

    def tensor_row(name, ms, flops):
        tf = flops / (ms * 1e-3) / 1e12
        return {"workload": name, "ms": ms, "value": tf, "unit": "TFLOP/s", "bound": "tensor",
                "frac": tf / bf16_peak}

    def hbm_row(name, ms, nbytes):
        gbs = nbytes / (ms * 1e-3) / 1e9
        return {"workload": name, "ms": ms, "value": gbs, "unit": "GB/s", "bound": "hbm", "frac": gbs / hbm_peak}

    rows = {}
    win, sinks = 4096, 4

    host = {}

    def llama_inputs():
        pc = workloads.config("llama3_8b")
        if "llama" not in host:  # drawn once on the CPU, copied to the device for each row
            host["llama"] = workloads.prefill_inputs(pc, seed=0)
        q, k, v = (t.to(dev) for t in host["llama"])
        return pc, q, k, v, torch.empty_like(q), torch.empty_like(k)

    def prefill_half_rope():  # split-halves RoPE pairing on the prefill workload
        pc, q, k, v, out, k_rot = llama_inputs()
        ms = timed(lambda: attn.prefill(q, k, v, rope_base=pc["rope_base"], scale=pc["scale"], out=out,
                                        k_rot=k_rot, pairing="half", stream=stream))
        return tensor_row("llama3-8b prefill B=4 S=8192, split-halves RoPE pairing", ms,
                          workloads.causal_flops(pc["B"], pc["S"], pc["n_h"], pc["D_h"]))

    def prefill_window():  # sliding window of 4096 keys plus 4 sinks on the prefill workload
        pc, q, k, v, out, k_rot = llama_inputs()
        ms = timed(lambda: attn.prefill_window(q, k, v, window=win, n_sink=sinks, rope_base=pc["rope_base"],
                                               scale=pc["scale"], out=out, k_rot=k_rot, stream=stream))
        return tensor_row(f"llama3-8b prefill B=4 S=8192, window {win} + {sinks} sinks", ms,
                          4.0 * pc["D_h"] * pc["n_h"] * pc["B"] * visible_pairs(range(pc["S"]), pc["S"], win, sinks))

    def prefill_chunk():  # the last 2048 queries at offset 6144 over the 8192-key rotated cache
        pc, q, k, v, out, k_rot = llama_inputs()
        attn.prefill(q, k, v, rope_base=pc["rope_base"], scale=pc["scale"], out=out, k_rot=k_rot, stream=stream)
        off, sq = 6144, 2048
        qc = q[:, off:].contiguous()
        outc = torch.empty_like(qc)
        ms = timed(lambda: attn.prefill_chunk(qc, k_rot, v, q_offset=off, rope_base=pc["rope_base"],
                                              scale=pc["scale"], out=outc, stream=stream))
        return tensor_row(f"llama3-8b chunk of {sq} queries at offset {off}, B=4, over an 8192-key cache", ms,
                          4.0 * pc["D_h"] * pc["n_h"] * pc["B"] * visible_pairs(range(off, off + sq), off + sq))

    def rope():  # the RoPE pass alone, on Q (268 MB in, 268 MB out)
        pc, q, _, _, qr, _ = llama_inputs()
        ms = timed(lambda: attn.rope(q, rope_base=pc["rope_base"], out=qr, stream=stream))
        return hbm_row("RoPE of llama3-8b Q [4,8192,32,128] bf16", ms, 2.0 * q.numel() * q.element_size())

    def kv_append():  # fused RoPE + KV append: an 8192-token prompt per sequence into a 16384-slot cache
        pc, _, k, v, _, _ = llama_inputs()
        B, S, n_kv, D = pc["B"], pc["S"], pc["n_kv"], pc["D_h"]
        kcache = torch.empty((B, 2 * S, n_kv, D), dtype=k.dtype, device=dev)
        vcache = torch.empty_like(kcache)
        start = torch.full((B,), 4096, dtype=torch.int32, device=dev)
        ms = timed(lambda: attn.kv_append(k, v, kcache, vcache, start, rope_base=pc["rope_base"], stream=stream))
        return hbm_row("append 8192 new tokens per sequence, B=4 n_kv=8 D=128, RoPE fused", ms,
                       2.0 * (k.numel() + v.numel()) * k.element_size())

    def decode_window():  # windowed GQA decode on the decode workload
        gc = workloads.config("gqa_decode")
        gq_h, gkc_h, gvc_h, gsl_h = workloads.decode_inputs(gc, seed=0)
        gq, gkc, gvc, gsl = gq_h.to(dev), gkc_h.to(dev), gvc_h.to(dev), gsl_h.to(dev)
        gws = torch.empty(attn.decode_workspace_size(gc["B"], gc["n_h"], gc["n_kv"], gc["D_qk"], gc["D_v"],
                                                     gc["max_len"]), dtype=torch.uint8, device=dev)
        gout = torch.empty(gc["B"], gc["n_h"], gc["D_v"], dtype=torch.bfloat16, device=dev)
        ms = timed(lambda: attn.decode_window(gq, gkc, gvc, gsl, window=win, n_sink=sinks,
                                              rope_base=gc["rope_base"], rope_dims=gc["rope_dims"],
                                              scale=gc["scale"], out=gout, workspace=gws, stream=stream))
        keys = sum(window_decode_keys(L, win, sinks) for L in gsl_h.tolist())
        return hbm_row(f"GQA decode 59 seqs L~U[4096,8192], window {win} + {sinks} sinks", ms,
                       keys * gc["n_kv"] * (gc["D_qk"] + gc["D_v"]) * 2.0)

    def decode_step(name):
        """One decode step: the new token's key (and value) appended to the cache at slot
        seqlens[b] - 1 (RoPE fused where the configuration rotates), then attention over the
        cache.  GB/s over the decode's cache bytes plus the append's bytes; the append alone
        is reported in microseconds."""
        cfg = workloads.config(name)
        q_h, kc_h, vc_h, sl_h = workloads.decode_inputs(cfg, seed=0)
        q, kc, sl = q_h.to(dev), kc_h.to(dev), sl_h.to(dev)
        alias = cfg.get("v_aliases_k")
        vc = kc[..., :cfg["D_v"]] if alias else vc_h.to(dev)
        g = torch.Generator().manual_seed(1)
        B, n_kv, D_qk, D_v = cfg["B"], cfg["n_kv"], cfg["D_qk"], cfg["D_v"]
        k_new = torch.randn((B, 1, n_kv, D_qk), generator=g).to(torch.bfloat16).to(dev)
        v_new = None if alias else torch.randn((B, 1, n_kv, D_v), generator=g).to(torch.bfloat16).to(dev)
        start = (sl - 1).to(torch.int32)
        ws = torch.empty(attn.decode_workspace_size(B, cfg["n_h"], n_kv, D_qk, D_v, cfg["max_len"]),
                         dtype=torch.uint8, device=dev)
        out = torch.empty(B, cfg["n_h"], D_v, dtype=torch.bfloat16, device=dev)
        rk = dict(rope_base=cfg["rope_base"], rope_offset=cfg["rope_offset"], rope_dims=cfg["rope_dims"])

        def append():
            attn.kv_append(k_new, v_new, kc, vc, start, stream=stream, **rk)

        def step():
            append()
            attn.decode(q, kc, vc, sl, scale=cfg["scale"], out=out, workspace=ws, stream=stream, **rk)

        ms_append = timed(append)
        ms = timed(step)
        new_bytes = 2.0 * B * n_kv * (D_qk + (0 if alias else D_v)) * 2  # read and written once
        row = hbm_row(f"{name} step: append 1 new token per sequence, then decode", ms,
                      workloads.decode_bytes(cfg, sl_h.tolist()) + new_bytes)
        row["kv_append_us"] = ms_append * 1e3
        return row

    def prefill_mla():  # MLA prefill on the non-absorbed path
        mc = workloads.config("mla_prefill")
        mq, mk, mv = (t.to(dev) for t in workloads.mla_prefill_inputs(mc, seed=0))
        mout, mk_rot = torch.empty_like(mv), torch.empty_like(mk)
        ms = timed(lambda: attn.prefill_mla(mq, mk, mv, rope_base=mc["rope_base"], rope_offset=mc["rope_offset"],
                                            rope_dims=mc["rope_dims"], scale=mc["scale"], out=mout, k_rot=mk_rot,
                                            stream=stream))
        return tensor_row("MLA prefill B=1 S=4096 128 heads, D_qk=192 D_v=128, RoPE on 64 dims", ms,
                          workloads.causal_flops(1, mc["S"], mc["n_h"], mc["D_qk"], mc["D_v"]))

    def prefill_gpt2():  # GPT-2-small-shaped prefill (D_h = 64, no RoPE)
        g2 = workloads.config("gpt2")
        q2, k2, v2 = (t.to(dev) for t in workloads.prefill_inputs(g2, seed=0))
        out2 = torch.empty_like(q2)
        ms = timed(lambda: attn.prefill(q2, k2, v2, scale=g2["scale"], out=out2, stream=stream))
        return tensor_row("GPT-2-small prefill B=8 S=1024 12 heads D=64", ms,
                          workloads.causal_flops(g2["B"], g2["S"], g2["n_h"], g2["D_h"]))

    table = [("prefill_half_rope", prefill_half_rope), ("prefill_window", prefill_window),
             ("prefill_chunk", prefill_chunk), ("rope", rope), ("kv_append", kv_append),
             ("decode_window", decode_window), ("decode_step_gqa", lambda: decode_step("gqa_decode")),
             ("decode_step_mla", lambda: decode_step("mla_decode")), ("prefill_mla", prefill_mla),
             ("prefill_gpt2", prefill_gpt2)]
    want = set(args.rows.split(",")) if args.rows else {name for name, _ in table}
    unknown = want - {name for name, _ in table}
    if unknown:
        raise SystemExit(f"unknown rows: {sorted(unknown)}")
    for name, fn in table:
        if name in want:
            rows[name] = fn()
            torch.cuda.empty_cache()

    line = {"impl": "ours", "extras": rows, "steps": args.steps, "warmup": args.warmup, "dtype": "bf16",
            "data": "synthetic", "l2": "256 MB flush write before every timed call",
            "peaks": {"bf16_tflops": bf16_peak, "hbm_gbs": hbm_peak, "source": peak_kind}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing")
    ap.add_argument("--parts", default="prefill,gqa,mla,gpt2",
                    help="comma-separated subset of prefill,gqa,mla,gpt2 (profiling runs)")
    ap.add_argument("--extras", action="store_true",
                    help="time the calls outside the default step instead (separate JSON line)")
    ap.add_argument("--rows", default="",
                    help="with --extras: comma-separated subset of its rows (profiling runs)")
    ap.add_argument("--prefill-batch", type=int, default=4,
                    help="batch of the prefill workload (4 = the benchmark workload; smaller for profiling)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("at least 3 warm-up steps")
    args.parts = [p for p in args.parts.split(",") if p]
    if args.impl == "reference":
        return run_reference(args)
    if args.extras:
        return run_extras(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
