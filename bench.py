#!/usr/bin/env python
"""Benchmark of the KDA layer step on GB300.

Headline workload (one bench step): KDA decode at batch 1, H = 64 heads,
d_k = d_v = 128, bf16 activations, fp32 state in a 256-slot pool, the state
warmed by 512 prior tokens; one step is 1000 chained decode launches
replayed from a CUDA graph.  value = decoded tokens / second.

Beside it the same JSON line carries the HBM roofline of the step kernel at
batch 64 (decode, and verify with T = 8 drafts) and the chunked prefill of
one 32768-token sequence; the CPU oracle is timed on the host cores as the
baseline.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch under torchrun; each rank runs an independent replica
(the layer step has no exchange between sequences), and value sums them.
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
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from hybrid_linear_attention_03_gb300 import inputs as I  # noqa: E402

METRIC = "KDA decode tok/s (batch 1, H=64, d=128, 1000 chained steps)"
UNIT = "tok/s"
STEP_KERNEL = "kda_step_kernel"
STEP_SOURCES = ("hybrid_linear_attention_03_gb300/csrc/kda_step.cu",
                "hybrid_linear_attention_03_gb300/csrc/kda_sm100.cuh",
                "hybrid_linear_attention_03_gb300/csrc/kda_internal.h")
L2_FLUSH_BYTES = 512 << 20
L2_NOTE = ("flushed before every timed launch: a 512 MiB buffer is written, then read, so the kernel "
           "finds none of its data in L2 and no dirty line of the flush is left for it to write back")


def flush_l2(buf):
    """Evicts L2 by writing a buffer 4x its size, then reading it back (the
    read makes the flush's own write-backs happen before the timed region)."""
    buf.zero_()
    return buf.view(torch.int64).sum()


def source_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


PREFILL_SOURCES = ("hybrid_linear_attention_03_gb300/csrc/kda_prefill.cu",
                   "hybrid_linear_attention_03_gb300/csrc/kda_prefill.cuh",
                   "hybrid_linear_attention_03_gb300/csrc/kda_prefill_intra_fast.cu",
                   "hybrid_linear_attention_03_gb300/csrc/kda_prefill_intra_generic.cu",
                   "hybrid_linear_attention_03_gb300/csrc/kda_sm100.cuh")
# Algorithmic FLOP per (chunk, head) at C = 64, d_k = d_v = 128 (full-square products):
# intra-chunk A, P, W, Ut (2 C^2 d each) and the triangular inverse (C^3 / 3);
# chain W S, Q S, K^T U (2 C d^2 each) and P U (2 C^2 d).
C_, D_ = 64, 128
INTRA_FLOP_PER_CHUNK_HEAD = 4 * 2 * C_ * C_ * D_ + C_ ** 3 // 3
CHAIN_FLOP_PER_CHUNK_HEAD = 3 * 2 * C_ * D_ * D_ + 2 * C_ * C_ * D_
# Algorithmic HBM bytes per prefill token at H = 64, d = 128, bf16: q, k, v, alpha, gate in, beta in, y out
PREFILL_BYTES_PER_TOKEN = 64 * (5 * 128 * 2 + 2 + 128 * 2)


def profiled_traffic(profile):
    """DRAM bytes per launch that an ncu summary under profiles/ records for
    the step kernel, or None if the kernel's sources changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", profile)) as f:
            text = f.read()
    except OSError:
        return None
    sha = re.search(r"^source_sha256_16: ([0-9a-f]{16})", text, re.M)
    tr = re.search(r"^traffic_bytes_per_launch: (\d+)", text, re.M)
    if not sha or not tr or sha.group(1) != source_sha(STEP_SOURCES):
        return None
    return int(tr.group(1))


def profiled_prefill_traffic(profile):
    """DRAM bytes per (chunk, head) that an ncu summary under profiles/
    records for the intra-chunk kernel (measured on a small case; traffic
    grows in proportion to the chunk-heads a launch processes), or None if
    the prefill sources changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", profile)) as f:
            text = f.read()
    except OSError:
        return None
    sha = re.search(r"^source_sha256_16: ([0-9a-f]{16})", text, re.M)
    tr = re.search(r"^traffic_bytes_per_chunk_head: (\d+)", text, re.M)
    if not sha or not tr or sha.group(1) != source_sha(PREFILL_SOURCES):
        return None
    return int(tr.group(1))


def args_():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the CPU oracle timing (profiling runs)")
    ap.add_argument("--only", choices=["decode_b64", "verify_b64_t8", "decode_b1_l2_flushed", "decode_b1_prefetch",
                                       "prefill", "mixed", "next_rows"], default=None,
                    help="run one secondary case alone (for profiling) and print its numbers")
    ap.add_argument("--prefill-tokens", type=int, default=None,
                    help="with --only prefill: a shorter sequence of the same workload (small profiling case)")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


# The layer has no exchange step: under torchrun every rank runs its own
# replica of the workload, and the ranks meet only around the timed region.
def settle(kda, stream, limit_s=300.0):
    """Waits for the stream with the library's watchdog (a bench that stops
    making progress fails with a message instead of hanging), then for the
    whole device."""
    if kda.kda_stream_wait(stream, limit_s) != kda.KDA_OK:
        raise RuntimeError(f"bench: the timed stream had not finished after {limit_s:.0f} s")
    torch.cuda.synchronize()


def rank_barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(ms, world, device):
    """The slowest rank's timed milliseconds (every rank holds the result)."""
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms):
    """Units all ranks processed per second over the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]),
                float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [int(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": float(statistics.median(sm)), "sm_max_mhz": float(max(int(r[2]) for r in rows)),
                "reasons": reasons, "samples": len(rows)}


def step_bytes(H, D, B, T, act_bytes=2):
    """Algorithmic HBM bytes of one step-kernel launch: each sequence reads
    its state and conv tail once and writes them T times (decode: in place),
    reads its T tokens' q, k, v, alpha, gate, beta, writes T outputs; conv
    weights and the norm weight are read once per launch."""
    state = H * D * D * 4
    tail = 3 * H * 3 * D * act_bytes
    io_tok = H * D * act_bytes * 5 + H * act_bytes + H * D * act_bytes
    weights = H * 3 * D * 4 * act_bytes + D * act_bytes
    return B * (state * (1 + T) + tail * (1 + T) + io_tok * T) + weights


# --------------------------------------------------------------------------- ours

def run_ours(a, rank, world, local):
    from hybrid_linear_attention_03_gb300 import build as kbuild
    from hybrid_linear_attention_03_gb300 import kda

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    hbm_peak, tf_peak, _, peak_kind = load_peaks()
    if a.only:
        kbuild.build()
        if a.only == "prefill":
            res = prefill_case(kda, dev, iters=a.steps, warmup=a.warmup, L=a.prefill_tokens)
        elif a.only == "next_rows":
            res = next_rows_case(kda, dev, iters=a.steps)
        elif a.only == "mixed":
            res = mixed_case(kda, dev, iters=a.steps, warmup=a.warmup)
        else:
            res = secondary(kda, dev, hbm_peak, peak_kind, only=a.only, iters=a.steps)
        print(json.dumps(res), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    kbuild.build()
    kda.lib()
    wl = I.DECODE_B1
    H, D, act, n_steps = wl.H, wl.dk, wl.act, wl.extra["steps"]

    w_cpu = wl.weights()
    w_dev = {k: v.to(dev) for k, v in w_cpu.items()}
    w = kda.make_weights(w_dev["conv_w"], w_dev["norm_w"], wl.eps_l2, wl.eps_rms)
    pool = kda.StatePool(wl.num_slots, H, D, D, act)
    slot = int(I.integers(wl.seed, 0, 0, wl.num_slots - 1, 1)[0])
    spare = (slot + 1) % wl.num_slots
    slot_t = torch.tensor([slot], dtype=torch.int32, device=dev)
    # warm the slot with 512 tokens (16 drafts per verify launch, the last one in place)
    warm = {k: v.to(dev) for k, v in wl.tokens(0, wl.extra["warm"]).items()}
    wout = torch.empty(16, H, D, dtype=act, device=dev)
    table = [s for s in range(wl.num_slots) if s not in (slot, spare)][:15] + [slot]
    snaps = torch.tensor(table, dtype=torch.int32, device=dev)
    for c in range(wl.extra["warm"] // 16):
        part = {k: v[c * 16:(c + 1) * 16] for k, v in warm.items()}
        kda.kda_verify(pool, w, kda.make_io(part, wout), slot_t, snaps, 1, 16)
    kda.kda_state_checkpoint(pool, [slot], [spare])  # the warm state, restored before every step
    torch.cuda.synchronize()

    toks = {k: v.to(dev) for k, v in wl.tokens(100, n_steps).items()}
    out = torch.empty(n_steps, H, D, dtype=act, device=dev)
    ios = [kda.make_io({k: v[i:i + 1] for k, v in toks.items()}, out[i:i + 1]) for i in range(n_steps)]
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        for i in range(3):  # first launches set kernel attributes, outside the capture
            kda.kda_decode(pool, w, ios[i], slot_t, 1)
        kda.kda_state_checkpoint(pool, [spare], [slot])
    stream.synchronize()
    # The chain's inputs are staged before it runs, so no kernel of the chain
    # writes a decode's inputs: the pool may let each launch fetch its inputs
    # under the previous launch (KDA_POOL_OVERLAP_INPUTS).  The same chain in
    # the default order (every read after the previous launch completes) is
    # timed beside it.
    graphs = {}
    for name, flags in (("overlap_inputs", kda.KDA_POOL_OVERLAP_INPUTS), ("default_order", 0)):
        kda.kda_state_pool_set_flags(pool, flags)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_steps):
                kda.kda_decode(pool, w, ios[i], slot_t, 1)
        graphs[name] = g
    kda.kda_state_pool_set_flags(pool, 0)
    graph = graphs["overlap_inputs"]

    def one_step(g=None):
        with torch.cuda.stream(stream):
            kda.kda_state_checkpoint(pool, [spare], [slot])
            flush_l2(flush)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            (g or graph).replay()
            e.record(stream)
        return s, e

    for _ in range(a.warmup):
        one_step()
    torch.cuda.synchronize()
    st, flags = kda.kda_poll_device_error(pool, stream)
    assert st == 0, f"device error word {flags:#x}"

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)
    rank_barrier(world)
    torch.cuda.synchronize()
    evs = [one_step() for _ in range(a.steps)]
    settle(kda, stream)
    rank_barrier(world)
    ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in evs), world, dev)
    value = job_throughput(a.steps * n_steps, world, ms)
    for _ in range(2):
        one_step(graphs["default_order"])
    evs_d = [one_step(graphs["default_order"]) for _ in range(a.steps)]
    settle(kda, stream)
    ms_d = max_over_ranks(sum(s.elapsed_time(e) for s, e in evs_d), world, dev)
    bytes_b1 = step_bytes(H, D, 1, 1)
    launch_us = ms * 1e3 / (a.steps * n_steps)
    achieved = bytes_b1 / (launch_us * 1e-6) / 1e9

    # end to end through the C ABI with host buffers: H2D of the step's inputs,
    # 1000 decodes, D2H of the outputs, all inside the timed region
    host_in = {k: v.pin_memory() for k, v in wl.tokens(100, n_steps).items()}
    host_out = torch.empty(n_steps, H, D, dtype=act).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        with torch.cuda.stream(stream):
            kda.kda_state_checkpoint(pool, [spare], [slot])
            flush_l2(flush)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            for k, v in host_in.items():
                toks[k].copy_(v, non_blocking=True)
            graph.replay()
            host_out.copy_(out, non_blocking=True)
            e.record(stream)
        return s, e

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    rank_barrier(world)
    evs2 = [e2e_step() for _ in range(a.steps)]
    settle(kda, stream)
    rank_barrier(world)
    ms2 = max_over_ranks(sum(s.elapsed_time(e) for s, e in evs2), world, dev)
    e2e_value = job_throughput(a.steps * n_steps, world, ms2)
    clk = clocks.stop()

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": round(ms / a.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy, value recipe of the workload)",
        "config": {"workload": wl.name, "batch": 1, "heads": H, "d_k": D, "d_v": D, "io_dtype": "bf16",
                   "state_dtype": "f32", "pool_slots": wl.num_slots, "warm_tokens": wl.extra["warm"],
                   "decode_steps_per_bench_step": n_steps, "cuda_graph": True,
                   "launch_order": "KDA_POOL_OVERLAP_INPUTS (inputs staged before the chain; each launch fetches "
                                   "them under the previous one)",
                   "l2": "flushed between timed steps (512 MiB written, then read); within a step the 4 MiB "
                         "state of the single sequence stays L2-resident across its 1000 chained decodes",
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": a.steps * n_steps,
        "roofline": {"bound": "hbm", "kernel": STEP_KERNEL, "achieved": round(achieved, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "traffic": profiled_traffic("kda_step_decode_b1_dram.md"),
                     "bytes_per_launch": bytes_b1, "launch_us": round(launch_us, 3),
                     "note": f"peak = {peak_kind} HBM copy bandwidth; at batch 1 the state stays in L2 and the "
                             "launch is latency-bound; the HBM rooflines of this kernel are the batch-64 entries "
                             "under secondary"},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "default_launch_order": {"value": round(job_throughput(a.steps * n_steps, world, ms_d), 1), "unit": UNIT,
                                 "launch_us": round(ms_d * 1e3 / (a.steps * n_steps), 3),
                                 "note": "the same chain with the pool's default launch order: each decode reads "
                                         "its inputs only after the previous launch has completed (what a caller "
                                         "whose inputs come from the kernel right before must use)"},
        "clocks": clk,
    }
    if not a.no_secondary:
        sec = secondary(kda, dev, hbm_peak, peak_kind)
        for name, fn in (("prefill", lambda: prefill_case(kda, dev, iters=3, warmup=1)),
                         ("mixed", lambda: mixed_case(kda, dev, iters=3, warmup=1)),
                         ("next_rows", lambda: next_rows_case(kda, dev))):
            try:
                sec[name] = fn()
            except Exception as e:  # reported, not hidden: the line says why the entry is absent
                sec[name] = {"error": f"{type(e).__name__}: {e}"}
            torch.cuda.empty_cache()
        line["secondary"] = sec
    if rank == 0:
        if not a.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(sample_tokens=n_steps)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def secondary(kda, dev, hbm_peak, peak_kind, only=None, iters=20):
    """HBM rooflines of the step kernel with L2 flushed before every launch:
    batch-64 decode (T = 1) and verify (T = 8), and a single batch-1 decode
    (its state then comes from HBM, unlike the chained headline steps)."""
    res = {}
    wl = I.VERIFY_B64
    H, D, act, B = wl.H, wl.dk, wl.act, wl.extra["B"]
    w_dev = {k: v.to(dev) for k, v in wl.weights().items()}
    w = kda.make_weights(w_dev["conv_w"], w_dev["norm_w"], wl.eps_l2, wl.eps_rms)
    pool = kda.StatePool(wl.num_slots, H, D, D, act)
    pool.states().normal_(0.0, 0.02)
    perm = torch.from_numpy(I.permutation(wl.seed, 0, wl.num_slots)).to(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for name, B, T, profile in (("decode_b64", wl.extra["B"], 1, "kda_step_decode_b64_full.md"),
                                ("verify_b64_t8", wl.extra["B"], 8, "kda_step_verify_b64_t8_dram.md"),
                                ("decode_b1_l2_flushed", 1, 1, "kda_step_decode_b1_cold_dram.md")):
        if only is not None and name != only:
            continue
        toks = {k: v.to(dev) for k, v in wl.tokens(200, B * T).items()}
        out = torch.empty(B * T, H, D, dtype=act, device=dev)
        io = kda.make_io(toks, out)
        snap = perm[:B * T].contiguous()
        ins = snap.view(B, T)[:, 0].contiguous()

        def launch():
            if T == 1:
                kda.kda_decode(pool, w, io, ins, B)
            else:
                kda.kda_verify(pool, w, io, ins, snap, B, T)

        for _ in range(3):
            launch()
        times = []
        for _ in range(iters):
            flush_l2(flush)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            launch()
            e.record(stream)
            e.synchronize()
            times.append(s.elapsed_time(e) * 1e3)
        us = float(np.mean(times))
        byts = step_bytes(H, D, B, T)
        ach = byts / (us * 1e-6) / 1e9
        res[name] = {"tok_per_s": round(B * T / (us * 1e-6), 1), "launch_us": round(us, 2),
                     "gpu_launches": iters,
                     "roofline": {"bound": "hbm", "kernel": STEP_KERNEL, "achieved": round(ach, 1),
                                  "peak": hbm_peak, "unit": "GB/s", "frac": round(ach / hbm_peak, 4),
                                  "traffic": profiled_traffic(profile), "bytes_per_launch": byts,
                                  "peak_kind": peak_kind},
                     "l2": L2_NOTE}
    # Batch-1 decodes inside a CUDA graph after other work of the layer.  Each
    # repetition of the graph runs [L2 flush] [kda_state_prefetch of n_seq
    # slots] a stand-in for the layer's other work (an element-wise op over 8
    # MiB the decodes do not touch, then copies that write their inputs the
    # way a projection would), then n_seq batch-1 decodes, each on its own
    # slot, so every decode after a flush finds its state in HBM.  A decode's
    # cost is the replay time with the decodes minus the same graph without
    # them, over the decodes, so the flush and the stand-in cancel.  Cases: L2
    # warm (no flush), L2 flushed, flushed with the slots prefetched before the
    # stand-in work, and with the slots and the layer weights.
    if only is None or only == "decode_b1_prefetch":
        n_seq, reps, replays = 16, 8, 4
        toks = {k: v.to(dev) for k, v in wl.tokens(210, n_seq).items()}
        src = {k: v.clone() for k, v in toks.items()}
        out = torch.empty(n_seq, H, D, dtype=act, device=dev)
        ios = [kda.make_io({k: v[i:i + 1] for k, v in toks.items()}, out[i:i + 1]) for i in range(n_seq)]
        slots = perm[:n_seq].contiguous()
        slot1 = [slots[i:i + 1] for i in range(n_seq)]
        busy_a = torch.ones(2 << 20, dtype=torch.float32, device=dev)
        busy_b = torch.empty_like(busy_a)
        gs = torch.cuda.Stream(device=dev)

        def body(flushed, pre, decode):
            for _ in range(reps):
                if flushed:
                    flush_l2(flush)
                if pre is not None:
                    kda.kda_state_prefetch(pool, slots, n_seq, weights=w if pre == "state+weights" else None)
                torch.mul(busy_a, 1.0001, out=busy_b)
                for k in toks:
                    toks[k].copy_(src[k])
                if decode:
                    for i in range(n_seq):
                        kda.kda_decode(pool, w, ios[i], slot1[i], 1)

        def replay_us(flushed, pre, decode):
            with torch.cuda.stream(gs):
                body(flushed, pre, decode)  # warm-up outside capture
            gs.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=gs):
                body(flushed, pre, decode)
            g.replay()
            torch.cuda.synchronize()
            st = torch.cuda.current_stream()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(st)
            for _ in range(replays):
                g.replay()
            e.record(st)
            e.synchronize()
            del g
            return s.elapsed_time(e) * 1e3 / replays

        res_p = {}
        for name, flushed, pre in (("l2_warm", False, None), ("l2_flushed", True, None),
                                   ("l2_flushed_state_prefetched", True, "state"),
                                   ("l2_flushed_state_weights_prefetched", True, "state+weights")):
            with_d = replay_us(flushed, pre, True)
            without = replay_us(flushed, pre, False)
            res_p[name] = {"decode_us": round((with_d - without) / (reps * n_seq), 2)}
        # the same decode as one event-timed launch outside a graph, after the
        # same stand-in work, with L2 warm and flushed: a spin with no memory
        # traffic first lets the host enqueue the rest, so no host gap is timed
        single = {}
        for name, flushed in (("l2_warm", False), ("l2_flushed", True)):
            times = []
            for _ in range(iters):
                if flushed:
                    flush_l2(flush)
                torch.cuda._sleep(400_000)
                torch.mul(busy_a, 1.0001, out=busy_b)
                for k in toks:
                    toks[k].copy_(src[k])
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record(stream)
                kda.kda_decode(pool, w, ios[0], slot1[0], 1)
                e.record(stream)
                e.synchronize()
                times.append(s.elapsed_time(e) * 1e3)
            single[name] = {"launch_us": round(float(np.mean(times)), 2)}
        res_p["single_launch"] = single
        res_p["note"] = (f"per batch-1 decode inside a CUDA graph: {n_seq} decodes on {n_seq} slots after an 8 MiB "
                         "element-wise op and copies writing their inputs (standing in for the layer's other work), "
                         f"{reps} repetitions per graph; replay time with the decodes minus without, over the "
                         "decodes; L2 flushed (512 MiB written, then read) before each repetition except in the "
                         "warm case; kda_state_prefetch of the slots issued before the stand-in work in the "
                         "prefetch cases; single_launch: one decode between two CUDA events after the same work, "
                         "outside a graph (launch latency included)")
        res["decode_b1_prefetch"] = res_p
    st, flags = kda.kda_poll_device_error(pool)
    assert st == 0, f"device error word {flags:#x}"
    return res


def prefill_case(kda, dev, iters=3, warmup=1, L=None):
    """Chunked prefill of one 32768-token sequence (H = 64, d = 128, C = 64,
    alpha = sigmoid(N(3, 1))) from a zero slot; tok/s of the whole call."""
    wl = I.PREFILL_32K
    H, D, act = wl.H, wl.dk, wl.act
    L = L or wl.extra["L"]
    w_dev = {k: v.to(dev) for k, v in wl.weights().items()}
    w = kda.make_weights(w_dev["conv_w"], w_dev["norm_w"], wl.eps_l2, wl.eps_rms)
    pool = kda.StatePool(wl.num_slots, H, D, D, act)
    toks = {k: v.to(dev) for k, v in wl.tokens(300, L).items()}
    out = torch.empty(L, H, D, dtype=act, device=dev)
    cu = [0, L]
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pool, cu), dtype=torch.uint8, device=dev)
    io = kda.make_io(toks, out)
    stream = torch.cuda.current_stream()

    def launch():
        kda.kda_prefill_chunked(pool, w, io, cu, [0], [0], 64, (), ws)

    for _ in range(warmup):
        launch()
    times = []
    for _ in range(iters):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        launch()
        e.record(stream)
        e.synchronize()
        times.append(s.elapsed_time(e))
    ms = float(np.mean(times))
    # one more call with the library's event profile: each kernel's device time
    # as it ran in the windowed schedule (events on the stream it launches on)
    kda.kda_profile_start(4096)
    launch()
    prof = kda.kda_profile_stop()
    st, flags = kda.kda_poll_device_error(pool)
    assert st == 0, f"device error word {flags:#x}"
    _, tf_peak, _, peak_kind = load_peaks()
    hbm_peak = load_peaks()[0]
    chunk_heads = ((L + 63) // 64) * H
    n_intra, intra_ms = prof["prefill_intra"]
    intra_flop = chunk_heads * INTRA_FLOP_PER_CHUNK_HEAD
    intra_tf = intra_flop / (intra_ms * 1e-3) / 1e12
    tr = profiled_prefill_traffic("kda_prefill_intra_fast_chain_4k_full.md")
    call_flop = chunk_heads * (INTRA_FLOP_PER_CHUNK_HEAD + CHAIN_FLOP_PER_CHUNK_HEAD)
    call_bytes = L * PREFILL_BYTES_PER_TOKEN
    return {"workload": wl.name if L == wl.extra["L"] else f"{wl.name} (first {L} tokens)",
            "tok_per_s": round(L / (ms / 1e3), 1), "ms_per_call": round(ms, 3),
            "workspace_bytes": ws.numel(),
            "kernels_ms_per_call": {k: round(v[1], 4) for k, v in prof.items() if k != "dropped" and v[0]},
            "kernel_launches_per_call": {k: v[0] for k, v in prof.items() if k != "dropped" and v[0]},
            "roofline": {"bound": "tensor", "kernel": "prefill_intra_fast_kernel", "achieved": round(intra_tf, 2),
                         "peak": tf_peak, "unit": "TFLOP/s", "frac": round(intra_tf / tf_peak, 4),
                         "traffic": None if tr is None else tr * chunk_heads // max(n_intra, 1),
                         "flop_per_launch": intra_flop // max(n_intra, 1),
                         "launch_us": round(intra_ms * 1e3 / max(n_intra, 1), 2),
                         "note": f"algorithmic intra-chunk FLOP (A, P, W, Ut and the triangular inverse: "
                                 f"{INTRA_FLOP_PER_CHUNK_HEAD} per chunk-head) over the factored-decay intra "
                                 f"kernel's device time, CUDA events around each of its launches inside the call "
                                 f"(one launch per window of chunks; the exact-decay kernel's hand-over list is "
                                 f"timed apart as prefill_intra_exact); peak = {peak_kind} dense bf16 (burst); "
                                 f"traffic = ncu DRAM bytes per chunk-head of a small case x the chunk-heads of "
                                 f"one launch"},
            "whole_call": {"algorithmic_flop": call_flop, "tflops": round(call_flop / (ms * 1e-3) / 1e12, 2),
                           "frac_bf16": round(call_flop / (ms * 1e-3) / 1e12 / tf_peak, 4),
                           "algorithmic_bytes": call_bytes, "gbs": round(call_bytes / (ms * 1e-3) / 1e9, 1),
                           "frac_hbm": round(call_bytes / (ms * 1e-3) / 1e9 / hbm_peak, 4)},
            "l2": "inputs (3.2 GB) exceed L2; not flushed between calls"}


def _event_us(stream, fn, iters):
    """Mean device time of fn() over iters calls, CUDA events on `stream`."""
    ts = []
    for _ in range(iters):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        fn()
        e.record(stream)
        e.synchronize()
        ts.append(s.elapsed_time(e) * 1e3)
    return float(np.mean(ts))


def next_rows_case(kda, dev, iters=20):
    """The widened rows, each measured: (1) prefill with device-built
    metadata in a CUDA graph against the host-built tables, for 1 and 64
    short sequences continuing their slots, and the same calls for new
    sequences (zero state); (2) the prefix cache: host planning time for a 32K-token
    prompt, and the GPU time of resuming from a saved prefix (slot copy plus
    the 64-token tail) against prefilling the whole prompt; (3) one slot's
    state export / import through pinned host memory."""
    wl = I.PREFILL_32K
    H, D, act = wl.H, wl.dk, wl.act
    w_dev = {k: v.to(dev) for k, v in wl.weights().items()}
    w = kda.make_weights(w_dev["conv_w"], w_dev["norm_w"], wl.eps_l2, wl.eps_rms)
    pool = kda.StatePool(160, H, D, D, act)
    stream = torch.cuda.Stream(device=dev)
    res = {}
    # (1) metadata: N sequences of 64 tokens each
    meta = {}
    for N in (1, 64):
        L = 64 * N
        toks = {k: v.to(dev) for k, v in wl.tokens(400, L).items()}
        out = torch.empty(L, H, D, dtype=act, device=dev)
        io = kda.make_io(toks, out)
        cu = np.arange(N + 1, dtype=np.int32) * 64
        slots, has = list(range(N)), [1] * N
        ws_h = torch.empty(kda.kda_prefill_workspace_bytes(pool, cu), dtype=torch.uint8, device=dev)
        cu_d = torch.tensor(cu, device=dev)
        sl_d = torch.tensor(slots, dtype=torch.int32, device=dev)
        hi_d = torch.tensor(has, dtype=torch.uint8, device=dev)
        ws_d = torch.empty(kda.kda_prefill_workspace_bytes_bound(pool, N, L, 0), dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            for _ in range(2):
                kda.kda_prefill_chunked(pool, w, io, cu, slots, has, 64, (), ws_h, stream)
                kda.kda_prefill_chunked_dev(pool, w, io, cu_d, sl_d, hi_d, L, None, ws_d, stream=stream)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            kda.kda_prefill_chunked_dev(pool, w, io, cu_d, sl_d, hi_d, L, None, ws_d, stream=stream)
        host_us = _event_us(stream, lambda: kda.kda_prefill_chunked(pool, w, io, cu, slots, has, 64, (), ws_h, stream),
                            iters)
        def replay():
            with torch.cuda.stream(stream):  # replay() launches on the current stream
                graph.replay()

        dev_us = _event_us(stream, replay, iters)
        # the same sequences started from a zero state: each is one chunk, which
        # the intra kernel finishes itself (the chain skips them)
        no_init = [0] * N
        new_us = _event_us(stream, lambda: kda.kda_prefill_chunked(pool, w, io, cu, slots, no_init, 64, (), ws_h, stream),
                           iters)
        # the metadata alone: the device builder kernel, against the host call's
        # table build (host wall time of the call, launches included) and the
        # device time of its tables' copies; library event profile
        kda.kda_profile_start(1024)
        for _ in range(iters):
            kda.kda_prefill_chunked_dev(pool, w, io, cu_d, sl_d, hi_d, L, None, ws_d, stream=stream)
        prof_dev = kda.kda_profile_stop()
        kda.kda_profile_start(1024)
        t0 = time.perf_counter()
        for _ in range(iters):
            kda.kda_prefill_chunked(pool, w, io, cu, slots, has, 64, (), ws_h, stream)
        host_call_us = (time.perf_counter() - t0) / iters * 1e6
        prof_host = kda.kda_profile_stop()
        stream.synchronize()
        meta[f"n{N}_x64_tokens"] = {
            "host_tables_us": round(host_us, 2), "device_tables_graph_us": round(dev_us, 2),
            "host_tables_new_sequences_us": round(new_us, 2),
            "meta_kernel_us": round(prof_dev["prefill_meta"][1] * 1e3 / max(prof_dev["prefill_meta"][0], 1), 2),
            "host_tables_copy_us": round(prof_host["prefill_meta"][1] * 1e3 / max(prof_host["prefill_meta"][0], 1),
                                         2),
            "host_call_wall_us": round(host_call_us, 2)}
        del graph
    res["device_metadata"] = meta
    # (2) prefix cache: a 32768-token prompt whose first 32704 tokens are saved
    L = wl.extra["L"]
    ids = [int(x) for x in I.integers(wl.seed, 7, 0, 1 << 30, L)]
    cache = kda.PrefixCache(64, [100], 1000)
    toks = {k: v.to(dev) for k, v in wl.tokens(300, L).items()}
    out = torch.empty(L, H, D, dtype=act, device=dev)
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pool, [0, L]), dtype=torch.uint8, device=dev)

    def full(reqs=()):
        kda.kda_prefill_chunked(pool, w, kda.make_io(toks, out), [0, L], [101], [0], 64, list(reqs), ws, stream)

    # a prompt of a whole number of blocks: its second plan admits the whole
    # prompt, which leaves no token to compute; the third admits one block
    # less, saved by that plan's prefill, and later plans reuse it
    plans = [cache.plan(ids) for _ in range(3)]
    _, _, admit_pos, admit_slot = plans[-1]
    with torch.cuda.stream(stream):
        full([(0, admit_pos, admit_slot)])
    ids_t = torch.tensor(ids, dtype=torch.int32)  # the token ids as one int32 array, as a server holds them
    t0 = time.perf_counter()
    n_plan = 20
    for _ in range(n_plan):
        hit, hit_slot, _, _ = cache.plan(ids_t)
    plan_us = (time.perf_counter() - t0) / n_plan * 1e6
    assert hit == admit_pos and hit_slot == admit_slot
    tail = {k: v[hit:].contiguous() for k, v in toks.items()}
    out_t = out[hit:]

    def resumed():
        kda.kda_state_checkpoint(pool, [hit_slot], [102], stream)
        kda.kda_prefill_chunked(pool, w, kda.make_io(tail, out_t), [0, L - hit], [102], [1], 64, (), ws, stream)

    with torch.cuda.stream(stream):
        full()
        resumed()
    stream.synchronize()
    res["prefix_cache"] = {"prompt_tokens": L, "reused_prefix_tokens": hit, "host_plan_us": round(plan_us, 1),
                           "full_prefill_us": round(_event_us(stream, full, 3), 1),
                           "copy_and_tail_prefill_us": round(_event_us(stream, resumed, iters), 1)}
    # (3) state export / import of one slot (state + conv tail) through pinned memory
    nb = kda.kda_state_slot_bytes(pool)
    host = torch.empty(nb, dtype=torch.uint8).pin_memory()
    ex_us = _event_us(stream, lambda: kda.kda_state_export(pool, 3, host, stream), iters)
    im_us = _event_us(stream, lambda: kda.kda_state_import(pool, 4, host, stream), iters)
    res["state_transfer"] = {"slot_bytes": nb, "export_us": round(ex_us, 1), "import_us": round(im_us, 1),
                             "export_gbs": round(nb / (ex_us * 1e-6) / 1e9, 1),
                             "import_gbs": round(nb / (im_us * 1e-6) / 1e9, 1)}
    st, flags = kda.kda_poll_device_error(pool, stream)
    assert st == 0, f"device error word {flags:#x}"
    return res


def mixed_case(kda, dev, iters=3, warmup=1):
    """The mixed step: one chunked-prefill call over 8 varlen sequences
    (log-uniform 1K..64K tokens, checkpoints every 32768 tokens and at each
    end into fresh slots) plus one decode call for 56 sequences warmed by 512
    tokens, over a 1024-slot pool.  tok/s = (prefill tokens + 56) / time."""
    wl = I.MIXED
    plan = I.mixed_plan(wl)
    H, D, act = wl.H, wl.dk, wl.act
    w_dev = {k: v.to(dev) for k, v in wl.weights().items()}
    w = kda.make_weights(w_dev["conv_w"], w_dev["norm_w"], wl.eps_l2, wl.eps_rms)
    pool = kda.StatePool(wl.num_slots, H, D, D, act)
    nd, warm_n, lens = wl.extra["n_decode"], wl.extra["warm"], plan["lens"]
    warm = {k: v.to(dev) for k, v in I.concat_inputs([wl.tokens(b, warm_n) for b in range(nd)]).items()}
    cu_w = [warm_n * i for i in range(nd + 1)]
    ws_w = torch.empty(kda.kda_prefill_workspace_bytes(pool, cu_w), dtype=torch.uint8, device=dev)
    wout = torch.empty(nd * warm_n, H, D, dtype=act, device=dev)
    kda.kda_prefill_chunked(pool, w, kda.make_io(warm, wout), cu_w, plan["dec_slots"], [0] * nd, 64, (), ws_w)
    del ws_w, wout, warm
    pf = {k: v.to(dev) for k, v in I.concat_inputs([wl.tokens(300 + n, L) for n, L in enumerate(lens)]).items()}
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pool, cu), dtype=torch.uint8, device=dev)
    out_pf = torch.empty(cu[-1], H, D, dtype=act, device=dev)
    dec = {k: v.to(dev) for k, v in wl.tokens(400, nd).items()}
    out_dec = torch.empty(nd, H, D, dtype=act, device=dev)
    dslots = torch.tensor(plan["dec_slots"], dtype=torch.int32, device=dev)
    io_pf, io_dec = kda.make_io(pf, out_pf), kda.make_io(dec, out_dec)
    stream = torch.cuda.current_stream()

    def step():
        kda.kda_prefill_chunked(pool, w, io_pf, cu, plan["pf_slots"], [0] * len(lens), 64, plan["reqs"], ws)
        kda.kda_decode(pool, w, io_dec, dslots, nd)

    for _ in range(warmup):
        step()
    times = []
    for _ in range(iters):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        step()
        e.record(stream)
        e.synchronize()
        times.append(s.elapsed_time(e))
    ms = float(np.mean(times))
    st, flags = kda.kda_poll_device_error(pool)
    assert st == 0, f"device error word {flags:#x}"
    n_tok = cu[-1] + nd
    return {"workload": wl.name, "tok_per_s": round(n_tok / (ms / 1e3), 1), "ms_per_step": round(ms, 3),
            "prefill_tokens": cu[-1], "decode_tokens": nd, "checkpoints": len(plan["reqs"]),
            "workspace_bytes": ws.numel()}


# ----------------------------------------------------------------------- oracle

def oracle_warm_state(o, wl, w):
    """The batch-1 sequence's state and conv tail after its 512 warm-up
    tokens, by the oracle: the start state of the timed decode steps, as in
    the GPU arm (which warms its slot with the same tokens)."""
    S = np.zeros((wl.H, wl.dk, wl.dv))
    tail = np.zeros((3, wl.H * (2 * wl.dk + wl.dv)))
    warm = {k: v.double().numpy() for k, v in wl.tokens(0, wl.extra["warm"]).items()}
    _, S, tail, _, _ = o.layer(warm, w, S, tail, eps_l2=wl.eps_l2, eps_rms=wl.eps_rms)
    return S, tail


def oracle_decode_run(o, wl, w, tok, n, start, n_threads=0):
    """The CPU oracle over n chained decode tokens of the batch-1 sequence,
    from the warm state `start`; returns the seconds it took."""
    S, tail = start
    part = {k: v[:n] for k, v in tok.items()}
    t0 = time.perf_counter()
    o.layer(part, w, S, tail, eps_l2=wl.eps_l2, eps_rms=wl.eps_rms, n_threads=n_threads)
    return time.perf_counter() - t0


def cpu_baseline(sample_tokens=1000, min_s=6.0, max_s=12.0):
    """The oracle as it stands on the host cores: chained batch-1 decode on
    all cores and on one thread (tok/s), and the 32K-token prefill's
    sequential token loop on a sample of heads and tokens, scaled to 64
    heads (tok/s).  A baseline, not the target."""
    from oracle import kda_oracle as ko

    o = ko.Oracle(ko.build())
    wl = I.DECODE_B1
    w = {k: v.double().numpy() for k, v in wl.weights().items()}
    tok = {k: v.double().numpy() for k, v in wl.tokens(100, sample_tokens).items()}
    start = oracle_warm_state(o, wl, w)
    total, n, runs = 0.0, 0, 0
    while total < min_s and runs < 100:
        total += oracle_decode_run(o, wl, w, tok, sample_tokens, start)
        n += sample_tokens
        runs += 1
        if total > max_s:
            break
    one_n = 100
    one_s = oracle_decode_run(o, wl, w, tok, one_n, start, n_threads=1)
    # prefill: the token loop (the oracle's definition) over the first L_s tokens of
    # H_s heads of the 32K-token workload; heads are independent, so the 64-head
    # rate is the sampled rate x H_s / 64
    pw = I.PREFILL_32K
    H_s, L_s = 16, 1024
    wp = {k: v.double().numpy() for k, v in pw.weights().items()}
    heads = list(range(H_s))
    chans = np.array([h * pw.dk + i for h in heads for i in range(pw.dk)] +
                     [pw.H * pw.dk + h * pw.dk + i for h in heads for i in range(pw.dk)] +
                     [2 * pw.H * pw.dk + h * pw.dv + j for h in heads for j in range(pw.dv)])
    ptok = {k: v[:, :H_s].double().numpy() for k, v in pw.tokens(300, L_s).items()}
    wps = {"conv_w": wp["conv_w"][chans], "norm_w": wp["norm_w"]}
    t0 = time.perf_counter()
    o.layer(ptok, wps, np.zeros((H_s, pw.dk, pw.dv)), np.zeros((3, H_s * (2 * pw.dk + pw.dv))),
            eps_l2=pw.eps_l2, eps_rms=pw.eps_rms)
    pf_s = time.perf_counter() - t0
    cores = o.max_threads()
    return {"value": round(n / total, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{runs} x {sample_tokens} chained decode tokens of the batch-1 workload from its 512-token "
                      f"warm state (float64 token loop, OpenMP over the 64 heads)",
            "one_thread": {"value": round(one_n / one_s, 2), "unit": UNIT, "cores": 1,
                           "sample": f"{one_n} chained decode tokens, one thread"},
            "prefill": {"value": round(L_s / pf_s * H_s / pw.H, 1), "unit": "tok/s", "cores": min(cores, H_s),
                        "sample": f"token loop over the first {L_s} tokens of {H_s} of the 64 heads of the "
                                  f"32768-token prefill workload, rate scaled by {H_s}/64 (heads are independent)"},
            "note": "CPU baseline, not the target"}


def run_reference(a, rank, world):
    if rank != 0:
        return
    from oracle import kda_oracle as ko

    o = ko.Oracle(ko.build())
    wl = I.DECODE_B1
    n = wl.extra["steps"]
    w = {k: v.double().numpy() for k, v in wl.weights().items()}
    tok = {k: v.double().numpy() for k, v in wl.tokens(100, n).items()}
    start = oracle_warm_state(o, wl, w)
    for _ in range(a.warmup):
        oracle_decode_run(o, wl, w, tok, n, start)
    total = sum(oracle_decode_run(o, wl, w, tok, n, start) for _ in range(a.steps))
    value = a.steps * n / total
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": 1,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(total * 1e3 / a.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded numpy, value recipe of the workload)",
            "config": {"workload": wl.name, "batch": 1, "heads": wl.H, "d_k": wl.dk, "d_v": wl.dv,
                       "warm_tokens": wl.extra["warm"], "decode_steps_per_bench_step": n},
            "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": o.max_threads(), "kind": "oracle",
                             "sample": f"{a.steps} x {n} chained decode tokens from the 512-token warm state "
                                       f"(the whole workload per step)"},
            "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    a = args_()
    rank, world, local = dist_env()
    if a.impl == "reference":
        run_reference(a, rank, world)
        return
    run_ours(a, rank, world, local)


if __name__ == "__main__":
    main()
