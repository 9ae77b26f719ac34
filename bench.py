"""Benchmark of the exact-attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
  attn_fwd           Qwen2.5-1.5B-style GQA prefill: B=4, Hq=12, Hkv=2,
                     N=4096, d=128, causal, bf16 (one launch)
  attn_decode_paged  64 sequences, Hq=12, Hkv=2, d=128, block_size 16,
                     lengths U[128, 4096], permuted block table (one launch;
                     seq_lens, the table and the cache come from host
                     copies, so the decode runs with its early plan at
                     level 2)
Also timed, outside the step and reported under their own keys:
  fwd_configs        attn_fwd on the GPT-2-small-shaped and long-context prefill
  backward           attn_bwd (dQ, dK, dV) on the Qwen-style prefill
  paged_prefill      attn_prefill_paged: 2048 new tokens per sequence on top of
                     a cached prefix of U[0, 6144] tokens (4 sequences,
                     Qwen-style GQA, block_size 16, permuted table)
  fusions            fused_add_rmsnorm and fused_swiglu on a Qwen2.5-1.5B-sized
                     layer over 16384 tokens (HBM GB/s)
  ssd                ssd_chunked_fwd (Mamba-2 SSD forward) on a Mamba-2-2.7B-
                     sized layer: batch 4, L 4096, 80 heads of 64, state 128
Printed (rank 0, one JSON line): fwd TFLOP/s as `value` (causal flops
4*B*Hq*N^2*d/2 over the forward kernel's CUDA-event time), the decode's HBM
GB/s under "decode" (algorithmic bytes over the time of decode calls run back
to back over the three rotated KV pools; the decode's time inside the step,
where it follows the forward's still-dirty output in L2, is reported beside
it), rooflines
against the measured peaks, the same metric end to end through the public
API with pinned host buffers ("e2e": every step uploads its inputs and reads
its results back; steps are pipelined over the three device sets with the
copies on two copy streams beside the compute stream, and the one-stream
figure is reported beside it), the fp64 oracle on host cores
("cpu_baseline"), and the SM clocks sampled while the GPU ran.

L2: three input sets (about 0.75 GB in total, above the 129 MB L2) are used
in rotation, so no step finds its inputs in L2 from the previous step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
Under torchrun (N > 1) every rank runs its own replica (its own seeds) with
no data exchange; times are max-reduced over ranks (weak scaling).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "attn fwd TFLOP/s (bf16, causal) & % tensor peak; paged-decode HBM GB/s"
FWD_CFG = "qwen_gqa_prefill"
DEC_CFG = "paged_decode"
NSETS = 3
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the bench step's
# kernels, from one single-kernel ncu capture of this workload (profiles/),
# valid only for the kernel source it was taken on: each entry keeps the
# sha256 of its source files at capture time, and bench reports the traffic
# as null once those files differ.
CSRC = os.path.join(ROOT, "exact_attention_47_gb300", "csrc")
TRAFFIC = {
    # median read + median write of 3 launches
    "fwd": {"bytes": 67196160 + 5156352, "sources": ("fwd_sm103.cu", "fwd_sm103.h", "ptx.cuh"),
            "sha256": "c061cce87aac37cddee53f431a14b87c1d506ad4be6b6457a2c5d3c8dc08a1fe"},
    # decode kernel (split parts merged inside it), median read + median write of 3 launches
    "dec": {"bytes": 132366848 + 414976, "sources": ("decode_sm103.cu", "decode_sm103.h", "ptx.cuh"),
            "sha256": "f99b6fe8bb0649fd0f754ee35830d2875c82b20eee2a8b35250d418badad3f9b"},
}


def source_digest(files):
    import hashlib

    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_for(key):
    """(bytes per launch or None, why) for a bench-step kernel."""
    rec = TRAFFIC[key]
    if rec["bytes"] is None or rec["sha256"] is None:
        return None, "not captured for this kernel source"
    if source_digest(rec["sources"]) != rec["sha256"]:
        return None, "kernel source changed since the capture"
    return rec["bytes"], "ncu capture of this kernel source (sha256 %s...)" % rec["sha256"][:12]


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def fwd_flops(c):
    return 4.0 * c["B"] * c["Hq"] * c["N"] * c["N"] * c["d"] / 2.0


def decode_bytes(inp, Hq, Hkv, d):
    total_L = int(inp["seq_lens"].to(torch.int64).sum())
    S = inp["q"].shape[0]
    kv = total_L * Hkv * d * 2 * 2                 # K and V rows addressed, bf16
    qo = S * Hq * d * 2 * 2                        # q in, o out
    lse = S * Hq * 4
    meta = S * inp["block_table"].shape[1] * 4 + S * 4
    return kv + qo + lse + meta


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.rows = []
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile(mode="w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                self.rows.append(dict(t=ts + frac, sm=float(parts[1]), sm_max=float(parts[2]),
                                      power=parts[3], active=parts[4], hw=parts[5], hwt=parts[6],
                                      swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        self.file.close()
        os.unlink(self.file.name)

    def summary(self, t0, t1):
        inside = [r for r in self.rows if t0 <= r["t"] <= t1]
        window = "timed region"
        if not inside:
            # the timed region was shorter than the sampling period: use the
            # samples of the busy period around it (warm-up + timed steps)
            inside = [r for r in self.rows if t0 - 1.0 <= r["t"] <= t1 + 1.0]
            window = "busy period around the timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        reasons = set()
        for r in inside:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["sm_max"] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


# ---------------------------------------------------------------- CPU arm

def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(target_s=12.0):
    """Time the fp64 oracle (as it stands) on whole (b, head) slices of the
    forward workload until about `target_s` seconds of CPU work are done."""
    import oracle

    c = workloads.PREFILL_CONFIGS[FWD_CFG]
    q, k, v = workloads.prefill_inputs(c["B"], c["Hq"], c["Hkv"], c["N"], c["d"], c["seed"])
    scale = workloads.default_scale(c["d"])
    qn, kn, vn = q.double().numpy(), k.double().numpy(), v.double().numpy()
    G = c["Hq"] // c["Hkv"]
    heads = 0
    t0 = time.perf_counter()
    while heads < c["B"] * c["Hq"]:
        b, h = divmod(heads, c["Hq"])
        oracle.attention(qn[b:b + 1, h:h + 1], kn[b:b + 1, h // G:h // G + 1],
                         vn[b:b + 1, h // G:h // G + 1], scale, True)
        heads += 1
        if time.perf_counter() - t0 >= target_s:
            break
    dt = time.perf_counter() - t0
    flops = 4.0 * heads * c["N"] * c["N"] * c["d"] / 2.0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": "%d of %d (batch, query head) slices of the %s workload (full causal rows), "
                      "fp64 numpy, %.1f s" % (heads, c["B"] * c["Hq"], FWD_CFG, dt)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle

    c = workloads.PREFILL_CONFIGS[FWD_CFG]
    q, k, v = workloads.prefill_inputs(c["B"], c["Hq"], c["Hkv"], c["N"], c["d"], c["seed"])
    scale = workloads.default_scale(c["d"])
    qn, kn, vn = q.double().numpy(), k.double().numpy(), v.double().numpy()
    G = c["Hq"] // c["Hkv"]

    def step(i):  # one (batch, head) slice of the forward workload per step
        b, h = divmod(i % (c["B"] * c["Hq"]), c["Hq"])
        oracle.attention(qn[b:b + 1, h:h + 1], kn[b:b + 1, h // G:h // G + 1],
                         vn[b:b + 1, h // G:h // G + 1], scale, True)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    flops = 4.0 * args.steps * c["N"] * c["N"] * c["d"] / 2.0
    value = flops / dt / 1e12
    sample = ("one (batch, query head) slice of the %s workload per step (N=%d, d=%d, causal), "
              "fp64 numpy oracle" % (FWD_CFG, c["N"], c["d"]))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": FWD_CFG + " (B4 Hq12 Hkv2 N4096 d128 causal)", "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def max_over_ranks(values, dist, device):
    """Each rank's timings -> the slowest rank's, on every rank."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_rates(world, steps, flops, dbytes, fwd_sum_ms, dec_sum_ms):
    """Whole-job forward TFLOP/s and decode GB/s (every rank runs the same
    work, timed by the slowest rank) and the per-GPU rates of one launch."""
    fwd_avg_s = fwd_sum_ms / steps / 1e3
    dec_avg_s = dec_sum_ms / steps / 1e3
    achieved_fwd = flops / fwd_avg_s / 1e12
    achieved_dec = dbytes / dec_avg_s / 1e9
    return world * achieved_fwd, world * achieved_dec, achieved_fwd, achieved_dec


def build_sets(rank, device):
    import exact_attention_47_gb300 as attn

    c = workloads.PREFILL_CONFIGS[FWD_CFG]
    dc = workloads.DECODE_CONFIGS[DEC_CFG]
    q, k, v = workloads.prefill_inputs(c["B"], c["Hq"], c["Hkv"], c["N"], c["d"],
                                       c["seed"] + 1000 * rank)
    dec = workloads.decode_inputs(dc["num_seqs"], dc["Hq"], dc["Hkv"], dc["d"],
                                  dc["seed"] + 1000 * rank, dc["len_lo"], dc["len_hi"])
    host = dict(q=q, k=k, v=v, dec=dec)
    sets = []
    ws_bytes = attn.attn_decode_paged_workspace_size(dc["num_seqs"], dc["Hq"], dc["d"],
                                                     dec["max_blocks_per_seq"])
    for _ in range(NSETS):
        s = dict(q=q.to(device), k=k.to(device), v=v.to(device),
                 o=torch.empty(q.shape, dtype=torch.bfloat16, device=device),
                 lse=torch.empty(q.shape[:3], dtype=torch.float32, device=device),
                 dq=dec["q"].to(device), kc=dec["k_cache"].to(device), vc=dec["v_cache"].to(device),
                 bt=dec["block_table"].to(device), sl=dec["seq_lens"].to(device),
                 do=torch.empty(dec["q"].shape, dtype=torch.bfloat16, device=device),
                 dlse=torch.empty(dec["q"].shape[:2], dtype=torch.float32, device=device),
                 ws=torch.empty(ws_bytes, dtype=torch.uint8, device=device))
        sets.append(s)
    return c, dc, host, sets


def decode_loop(attn, sets, scale, steps):
    """attn_decode_paged alone, back to back over the rotated input sets
    (three KV pools of about 140 MB: no call finds its cache in L2), CUDA
    events around the whole loop.  Returns ms per call (decode kernel and
    launch gaps included)."""
    def dec(s):
        attn.attn_decode_paged(s["dq"], s["kc"], s["vc"], s["bt"], s["sl"], scale=scale,
                               o=s["do"], lse=s["dlse"], workspace=s["ws"])

    for i in range(3 * len(sets)):
        dec(sets[i % len(sets)])
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        dec(sets[i % len(sets)])
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def fwd_config_table(attn, device, steps, peak):
    """Forward TFLOP/s on the other prefill configs (GPT-2-small-shaped, d = 64;
    long context, N = 16384), timed like the main workload: CUDA events over
    `steps` launches after 3 warm-ups, input sets rotated so that they exceed L2."""
    out = {}
    for name in ("gpt2_small", "long_context"):
        c = workloads.PREFILL_CONFIGS[name]
        nsets = 3 if name == "gpt2_small" else 1    # 3 x 50 MB, or one 268 MB set: > L2 either way
        sets = []
        for i in range(nsets):
            q, k, v = workloads.prefill_inputs(c["B"], c["Hq"], c["Hkv"], c["N"], c["d"], c["seed"] + 100 * i,
                                               std=c["std"], key_offset=c["key_offset"])
            sets.append((q.to(device), k.to(device), v.to(device)))
        scale = workloads.default_scale(c["d"])
        o = torch.empty_like(sets[0][0])
        lse = torch.empty(sets[0][0].shape[:3], dtype=torch.float32, device=device)
        for i in range(3):
            attn.attn_fwd(*sets[i % nsets], causal=True, scale=scale, o=o, lse=lse)
        stream = torch.cuda.current_stream()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(steps):
            attn.attn_fwd(*sets[i % nsets], causal=True, scale=scale, o=o, lse=lse)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        tflops = fwd_flops(c) / (ms / 1e3) / 1e12
        out[name] = {"shape": "B%d Hq%d Hkv%d N%d d%d causal" % (c["B"], c["Hq"], c["Hkv"], c["N"], c["d"]),
                     "ms": ms, "tflops": tflops, "frac": tflops / peak}
        del sets, o, lse
    return out


def bwd_measurement(attn, device, steps, peak):
    """attn_bwd on the qwen_gqa_prefill workload (both kernels per call),
    CUDA events over `steps` calls after 3 warm-ups.  FLOPs: 2.5 x the forward
    count (five matmuls of the forward's tile sizes against its two)."""
    c = workloads.PREFILL_CONFIGS[FWD_CFG]
    q, k, v = workloads.prefill_inputs(c["B"], c["Hq"], c["Hkv"], c["N"], c["d"], c["seed"])
    g = torch.Generator().manual_seed(c["seed"] + 5)
    do = torch.randn(q.shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    q, k, v, do = (t.to(device) for t in (q, k, v, do))
    scale = workloads.default_scale(c["d"])
    o, lse = attn.attn_fwd(q, k, v, causal=True, scale=scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(attn.attn_bwd_workspace_size(c["B"], c["Hq"], c["N"]), dtype=torch.uint8, device=device)
    for _ in range(3):
        attn.attn_bwd(q, k, v, o, lse, do, causal=True, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws)
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        attn.attn_bwd(q, k, v, o, lse, do, causal=True, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    tflops = 2.5 * fwd_flops(c) / (ms / 1e3) / 1e12
    return {"workload": FWD_CFG + " (B4 Hq12 Hkv2 N4096 d128 causal)", "ms": ms, "tflops": tflops,
            "frac": tflops / peak, "flop_convention": "2.5 x forward (5 matmuls vs 2)",
            "kernels": "rowdot + one grid of dK/dV and dQ tiles"}


def paged_prefill_flops(ctx_lens, Hq, N, d):
    """Causal pairs of a chunk: new query i sees ctx + i + 1 keys."""
    pairs = sum(N * int(c) + N * (N + 1) // 2 for c in ctx_lens)
    return 4.0 * d * Hq * pairs


def paged_prefill_measurement(attn, device, steps, peak):
    """attn_prefill_paged on the chunked-prefill workload (2048 new tokens on
    top of a cached prefix of U[0, 6144] tokens, 4 sequences, Qwen-style GQA,
    block_size 16, permuted table): the append and the attention kernel per
    call, CUDA events over `steps` calls after 3 warm-ups, three input sets
    (about 60 MB each) in rotation so they exceed L2.  Appending the same rows
    at the same positions again leaves the cache as it was, so every call does
    the same work."""
    c = workloads.PAGED_PREFILL_CONFIGS["qwen_chunked_prefill"]
    sets, flops = [], []
    for i in range(3):
        x = workloads.paged_prefill_inputs(c["num_seqs"], c["Hq"], c["Hkv"], c["N_new"], c["d"],
                                           c["seed"] + 100 * i, ctx_lo=c["ctx_lo"], ctx_hi=c["ctx_hi"])
        flops.append(paged_prefill_flops(x["ctx_lens"].tolist(), c["Hq"], c["N_new"], c["d"]))
        d = {n: x[n].to(device) for n in ("q", "k_new", "v_new", "k_cache", "v_cache",
                                          "block_table", "ctx_lens")}
        d["o"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(d["q"].shape[:3], dtype=torch.float32, device=device)
        sets.append(d)
    scale = workloads.default_scale(c["d"])

    def call(d):
        attn.attn_prefill_paged(d["q"], d["k_new"], d["v_new"], d["k_cache"], d["v_cache"],
                                d["block_table"], d["ctx_lens"], scale=scale, o=d["o"], lse=d["lse"])

    for i in range(3):
        call(sets[i % 3])
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        call(sets[i % 3])
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    mean_flops = sum(flops[i % 3] for i in range(steps)) / steps
    tflops = mean_flops / (ms / 1e3) / 1e12
    return {"workload": "qwen_chunked_prefill (4 seqs, N_new 2048, ctx~U[0,6144], Hq12 Hkv2 d128, "
                        "block_size 16)", "ms": ms, "tflops": tflops, "frac": tflops / peak,
            "flop_convention": "4*d*Hq*sum_b(N*ctx_b + N(N+1)/2) (causal pairs)",
            "kernels": "kv append + attention (paged mode)", "gpu_launches_per_call": 2}


def fusion_bytes(rows, hidden, F):
    """Algorithmic bytes of one call: add + RMSNorm reads x and residual and
    writes residual and out (plus the weight once); SwiGLU reads [rows, 2F]
    and writes [rows, F]; bf16 throughout."""
    return {"add_rmsnorm": 4 * rows * hidden * 2 + hidden * 2, "swiglu": 3 * rows * F * 2}


def ssd_flops(batch, L, H, G, P, N, chunk):
    """FLOPs of the chunked SSD forward per call, by the matrix form: per
    chunk of n positions, C B^T under the causal mask once per B/C group
    (n^2/2 pairs of N multiply-adds: n^2 N), and per head its product with X
    (n^2 P), the state update (x o w)^T B and the carried state's output
    C S^T (2 n P N each)."""
    total = 0
    for c0 in range(0, L, chunk):
        n = min(chunk, L - c0)
        total += G * n * n * N + H * (n * n * P + 4 * n * P * N)
    return float(batch * total)


def ssd_bytes(batch, L, H, G, P, N):
    """Algorithmic bytes per call: x, B, C (bf16), dt (fp32) and A read; y
    (bf16) and the final state (fp32) written."""
    return (batch * L * H * P * 2 + 2 * batch * L * G * N * 2 + batch * L * H * 4 + H * 4
            + batch * L * H * P * 2 + batch * H * P * N * 4)


def ssd_measurement(attn, device, steps, peak_tflops, peak_gbs):
    """ssd_chunked_fwd on the mamba2_ssd workload (x and y are 168 MB each,
    beyond L2), CUDA events over `steps` calls after 3 warm-ups.  Reported
    against both rooflines; its intensity sits near the ridge."""
    c = workloads.SSD_CONFIGS["mamba2_ssd"]
    d = workloads.ssd_inputs(c["batch"], c["L"], c["H"], c["P"], c["N"], c["G"], c["seed"])
    d = {k: v.to(device) for k, v in d.items()}
    y = torch.empty_like(d["x"])
    hf = torch.empty((c["batch"], c["H"], c["P"], c["N"]), dtype=torch.float32, device=device)
    ws = torch.empty(attn.ssd_workspace_size(c["batch"], c["L"], c["H"], c["N"], c["chunk"]),
                     dtype=torch.uint8, device=device)

    def call():
        attn.ssd_chunked_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], chunk=c["chunk"], y=y,
                             h_final=hf, workspace=ws)

    for _ in range(3):
        call()
    stream = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    flops = ssd_flops(c["batch"], c["L"], c["H"], c["G"], c["P"], c["N"], c["chunk"])
    nbytes = ssd_bytes(c["batch"], c["L"], c["H"], c["G"], c["P"], c["N"])
    tflops = flops / (ms / 1e3) / 1e12
    gbs = nbytes / (ms / 1e3) / 1e9
    bound = "tensor" if flops / peak_tflops / 1e12 >= nbytes / peak_gbs / 1e9 else "hbm"
    del d, y, hf, ws
    return {"workload": "mamba2_ssd (batch 4, L 4096, H 80, P 64, N 128, G 1, chunk 256)", "ms": ms,
            "tflops": tflops, "frac_tensor": tflops / peak_tflops, "GB/s": gbs, "frac_hbm": gbs / peak_gbs,
            "bound": bound, "flops": flops, "bytes": nbytes,
            "flop_convention": "per chunk of n: G n^2 N + H (n^2 P + 4 n P N) (causal pairs n^2/2)",
            "kernels": "chunk state (cumsum + fwd_pass_state) + chunk output", "gpu_launches_per_call": 2}


def swiglu_projection_flops(rows, hidden, F):
    """FLOPs of the gate/up projection: a [rows, hidden] x [hidden, 2F]
    product (the activation's few operations per output are not counted)."""
    return 2.0 * rows * 2 * F * hidden


def fusion_measurement(attn, device, steps, peak_gbs, peak_tflops):
    """fused_add_rmsnorm and fused_swiglu on one Qwen2.5-1.5B-sized layer over
    the 16384 prefill tokens (hidden 1536, intermediate 8960), CUDA events over
    `steps` calls after 3 warm-ups.  Algorithmic bytes: every input read once,
    every output written once (add + RMSNorm: x, residual in; residual, out
    out; swiglu: [rows, 2F] in, [rows, F] out).  Two input sets alternate for
    add + RMSNorm (2 x 151 MB > L2); one swiglu call moves 881 MB."""
    c = workloads.FUSION_CONFIGS["qwen_add_rmsnorm"]
    sets = []
    for i in range(2):
        x, res, w = workloads.add_rmsnorm_inputs(c["rows"], c["hidden"], c["seed"] + 100 * i)
        sets.append((x.to(device), res.to(device), w.to(device), torch.empty_like(x, device=device)))
    nbytes = fusion_bytes(c["rows"], c["hidden"], 0)["add_rmsnorm"]
    stream = torch.cuda.current_stream()

    def timed(fn, n):
        for i in range(3):
            fn(i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    ms_norm = timed(lambda i: attn.fused_add_rmsnorm(sets[i % 2][0], sets[i % 2][1], sets[i % 2][2],
                                                     out=sets[i % 2][3]), steps)
    del sets
    g = workloads.FUSION_CONFIGS["qwen_swiglu"]
    gu = workloads.swiglu_inputs(g["rows"], g["F"], g["seed"]).to(device)
    out = torch.empty((g["rows"], g["F"]), dtype=torch.bfloat16, device=device)
    gbytes = fusion_bytes(g["rows"], 0, g["F"])["swiglu"]
    ms_glu = timed(lambda i: attn.fused_swiglu(gu, out=out), steps)
    del gu, out
    res = {}
    for name, ms, b, shape in (("add_rmsnorm", ms_norm, nbytes, "rows 16384 hidden 1536"),
                               ("swiglu", ms_glu, gbytes, "rows 16384 F 8960")):
        gbs = b / (ms / 1e3) / 1e9
        res[name] = {"shape": shape, "ms": ms, "bytes": b, "GB/s": gbs, "frac": gbs / peak_gbs,
                     "bound": "hbm"}
    # The gate/up projection with the activation in its epilogue, beside the
    # unfused pair it replaces (a library GEMM writing [rows, 2F], then the
    # activation kernel): the library GEMM is a comparison point only.
    p = workloads.FUSION_CONFIGS["qwen_swiglu_projection"]
    x, w = workloads.swiglu_projection_inputs(p["rows"], p["hidden"], p["F"], p["seed"])
    x, w = x.to(device), w.to(device)
    out = torch.empty((p["rows"], p["F"]), dtype=torch.bfloat16, device=device)
    ms_proj = timed(lambda i: attn.swiglu_projection(x, w, out=out), steps)
    gu = torch.empty((p["rows"], 2 * p["F"]), dtype=torch.bfloat16, device=device)
    ms_unfused = timed(lambda i: (torch.matmul(x, w.T, out=gu), attn.fused_swiglu(gu, out=out)), steps)
    del x, w, out, gu
    pf = swiglu_projection_flops(p["rows"], p["hidden"], p["F"])
    tf = pf / (ms_proj / 1e3) / 1e12
    res["swiglu_projection"] = {"shape": "rows 16384 hidden 1536 F 8960", "ms": ms_proj, "flops": pf,
                                "TFLOP/s": tf, "frac": tf / peak_tflops, "bound": "tensor",
                                "unfused_library_gemm_plus_activation_ms": ms_unfused}
    return res


def run_gpu(args, rank, world, local_rank):
    import exact_attention_47_gb300 as attn

    # Every decode here reads seq_lens, a block table and a KV cache written
    # by host copies made before the step, never by the kernel just before
    # it (another decode or the forward, which write only their outputs), so
    # the plan and the first cache blocks may be read before that kernel
    # has finished (level 2).
    attn.set_decode_early_plan(2)
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    c, dc, host, sets = build_sets(rank, device)
    scale_f = workloads.default_scale(c["d"])
    scale_d = workloads.default_scale(dc["d"])
    flops = fwd_flops(c)
    dbytes = decode_bytes(host["dec"], dc["Hq"], dc["Hkv"], dc["d"])
    stream = torch.cuda.current_stream()

    def fwd(s):
        attn.attn_fwd(s["q"], s["k"], s["v"], causal=True, scale=scale_f, o=s["o"], lse=s["lse"])

    def dec(s):
        attn.attn_decode_paged(s["dq"], s["kc"], s["vc"], s["bt"], s["sl"], scale=scale_d,
                               o=s["do"], lse=s["dlse"], workspace=s["ws"])

    clock = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ
                         else os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank])
    clock.start()
    for i in range(args.warmup):
        s = sets[i % NSETS]
        fwd(s)
        dec(s)
    torch.cuda.synchronize()
    if attn.device_status() != 0:
        raise RuntimeError("device status flags set during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.time()
    t_start.record(stream)
    for i in range(K):
        s = sets[i % NSETS]
        ev[i][0].record(stream)
        fwd(s)
        ev[i][1].record(stream)
        dec(s)
        ev[i][2].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if dist:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[1].elapsed_time(e[2]) for e in ev]
    if attn.device_status() != 0:
        raise RuntimeError("device status flags set during the timed steps")

    # ---- end to end through the public API with pinned host buffers
    h_q, h_k, h_v = (host[x].pin_memory() for x in ("q", "k", "v"))
    hd = host["dec"]
    h_dq, h_bt, h_sl = hd["q"].pin_memory(), hd["block_table"].pin_memory(), hd["seq_lens"].pin_memory()
    # One set of pinned result buffers per device input set, so the read-backs
    # of consecutive steps never share a host buffer.
    h_out = [dict(o=torch.empty(h_q.shape, dtype=torch.bfloat16).pin_memory(),
                  lse=torch.empty(h_q.shape[:3], dtype=torch.float32).pin_memory(),
                  do=torch.empty(h_dq.shape, dtype=torch.bfloat16).pin_memory(),
                  dlse=torch.empty(h_dq.shape[:2], dtype=torch.float32).pin_memory()) for _ in range(NSETS)]
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_k, h_v, h_dq, h_bt, h_sl))
    d2h = sum(t.numel() * t.element_size() for t in h_out[0].values())

    def upload(s):
        s["q"].copy_(h_q, non_blocking=True)
        s["k"].copy_(h_k, non_blocking=True)
        s["v"].copy_(h_v, non_blocking=True)
        s["dq"].copy_(h_dq, non_blocking=True)
        s["bt"].copy_(h_bt, non_blocking=True)
        s["sl"].copy_(h_sl, non_blocking=True)

    def download(s, ho):
        ho["o"].copy_(s["o"], non_blocking=True)
        ho["lse"].copy_(s["lse"], non_blocking=True)
        ho["do"].copy_(s["do"], non_blocking=True)
        ho["dlse"].copy_(s["dlse"], non_blocking=True)

    def e2e_serial_step(i):
        s = sets[i % NSETS]
        upload(s)
        fwd(s)
        dec(s)
        download(s, h_out[i % NSETS])

    # Pipelined: step i's uploads run on one copy stream while the kernels of
    # step i - 1 run, and its read-backs on another; a device set is uploaded
    # again only once the read-back of the step that last used it is done.
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    set_free = [None] * NSETS

    def e2e_step(i):
        j = i % NSETS
        s = sets[j]
        if set_free[j] is not None:
            up.wait_event(set_free[j])
        with torch.cuda.stream(up):
            upload(s)
        inputs_in = torch.cuda.Event()
        inputs_in.record(up)
        stream.wait_event(inputs_in)
        fwd(s)
        dec(s)
        results = torch.cuda.Event()
        results.record(stream)
        down.wait_event(results)
        with torch.cuda.stream(down):
            download(s, h_out[j])
        set_free[j] = torch.cuda.Event()
        set_free[j].record(down)

    def timed_e2e(step, n):
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        up.wait_event(e0)
        down.wait_event(e0)
        for i in range(n):
            step(i)
        stream.wait_stream(up)
        stream.wait_stream(down)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    for i in range(max(1, min(args.warmup, 3))):
        e2e_step(i)
    e2e_ms = timed_e2e(e2e_step, K)
    # Every step's read-back is complete: the last step's results equal the
    # device outputs they were copied from.
    last = (K - 1) % NSETS
    e2e_ok = bool(torch.equal(h_out[last]["o"], sets[last]["o"].cpu()) and
                  torch.equal(h_out[last]["dlse"], sets[last]["dlse"].cpu()))
    e2e_serial_ms = timed_e2e(e2e_serial_step, max(50, K // 10))
    clock.stop()
    pk_all, _ = peaks()
    side = max(10, min(K, 200))      # calls per measurement outside the step
    dec_alone_ms = decode_loop(attn, sets, scale_d, max(200, K // 3))
    fwd_configs = fwd_config_table(attn, device, side, pk_all["bf16_tflops"])
    backward = bwd_measurement(attn, device, side, pk_all["bf16_tflops"])
    paged_prefill = paged_prefill_measurement(attn, device, side, pk_all["bf16_tflops"])
    fusions = fusion_measurement(attn, device, side, pk_all["hbm_gbs"], pk_all["bf16_tflops"])
    ssd = ssd_measurement(attn, device, side, pk_all["bf16_tflops"], pk_all["hbm_gbs"])

    # ---- max over ranks
    total_ms, fwd_sum, dec_sum, e2e_ms, dec_alone_ms, e2e_serial_ms = max_over_ranks(
        [total_ms, sum(fwd_ms), sum(dec_ms), e2e_ms, dec_alone_ms, e2e_serial_ms], dist, device)

    if rank == 0:
        pk, pk_kind = peaks()
        tflops, gbs_step, achieved_fwd, achieved_dec_step = job_rates(world, K, flops, dbytes, fwd_sum, dec_sum)
        achieved_dec = dbytes / (dec_alone_ms / 1e3) / 1e9
        gbs = world * achieved_dec
        clocks = clock.summary(wall0, wall1)
        traffic_fwd, traffic_fwd_src = traffic_for("fwd")
        traffic_dec, traffic_dec_src = traffic_for("dec")
        # time x median SM clock (ms x MHz = thousands of SM cycles): comparable
        # across runs whose clocks differ
        kcyc = (lambda ms: None if clocks.get("sm_mhz") is None else ms * clocks["sm_mhz"])
        line = {
            "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
            "kcycles_per_step": kcyc(total_ms / K),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "%s (B4 Hq12 Hkv2 N4096 d128 causal) + %s (64 seqs, Hq12 "
                                   "Hkv2 d128, block_size 16, L~U[128,4096])" % (FWD_CFG, DEC_CFG),
                       "l2": "3 input sets rotated (~0.75 GB > 129 MB L2); no flush",
                       "flop_convention": "4*B*Hq*N^2*d/2 (causal)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "roofline": {"bound": "tensor", "achieved": achieved_fwd,
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": achieved_fwd / pk["bf16_tflops"], "traffic": traffic_fwd,
                         "traffic_source": traffic_fwd_src,
                         "kcycles_per_launch": kcyc(fwd_sum / K),
                         "kernel": "attn_fwd_sm103_kernel<128,causal>",
                         "peak_kind": pk_kind + " burst bf16 (cuBLAS)",
                         "fwd_ms_mean": fwd_sum / K, "fwd_ms_median": statistics.median(fwd_ms)},
            "decode": {"value": gbs, "unit": "GB/s", "ms_mean": dec_alone_ms,
                       "bytes_per_step": dbytes,
                       "measured": "decode calls back to back over the 3 rotated KV pools (one kernel "
                                   "per call, launch gaps included), CUDA events around the loop",
                       "early_plan": "2: the split plan and each CTA's first 21 cache blocks (not a "
                                     "sequence's last) are read before the preceding kernel ends",
                       "in_step_ms_mean": dec_sum / K, "in_step_ms_median": statistics.median(dec_ms),
                       "in_step_GB/s": world * achieved_dec_step,
                       "in_step_note": "inside the step the decode follows the forward, whose 50 MB "
                                       "output is still dirty in L2; its write-back shares HBM with "
                                       "the decode's reads",
                       "roofline": {"bound": "hbm", "achieved": achieved_dec,
                                    "peak": pk["hbm_gbs"], "unit": "GB/s",
                                    "frac": achieved_dec / pk["hbm_gbs"], "traffic": traffic_dec,
                                    "traffic_source": traffic_dec_src,
                                    "kernel": "attn_decode_paged_kernel<128>",
                                    "peak_kind": pk_kind + " copy bandwidth"}},
            "e2e": {"value": world * flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "note": "fwd flops over the whole step: pinned h2d of q,k,v and of the "
                            "decode query/table/lengths, both ops, d2h of all outputs; steps "
                            "pipelined over the 3 device sets (uploads and read-backs on two copy "
                            "streams beside the compute stream)",
                    "readback_matches_device": e2e_ok,
                    "serial": {"value": world * flops / (e2e_serial_ms / 1e3) / 1e12,
                               "ms_per_step": e2e_serial_ms,
                               "note": "the same step with copies and kernels in one stream"}},
            "fwd_configs": dict(fwd_configs, **{FWD_CFG: {
                "shape": "B4 Hq12 Hkv2 N4096 d128 causal", "ms": fwd_sum / K,
                "tflops": achieved_fwd, "frac": achieved_fwd / pk["bf16_tflops"]}}),
            "backward": backward,
            "paged_prefill": paged_prefill,
            "fusions": fusions,
            "ssd": ssd,
            "gpu_launches": 2 * K,
            "timed_region_s": total_ms / 1e3,
            "clocks": clocks,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = oracle_sample(args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=6000)     # about 1.4 s of GPU time
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
