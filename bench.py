"""Benchmark of the layer-wise KV sparsification hot path on one GB300.

Workload: Llama-3-8B attention shapes, one request of 4000 prompt tokens and
500 generated tokens (32 layers, 32 query / 8 KV heads, d = 128, bf16;
layers 0-2 full cache, layers 3-31 budgets 2048 .. 256 incl. the 32 most
recent tokens, window alpha = 32), seeded synthetic inputs.

One bench step = one request through the whole hot path:
  prefill+sparsify  per layer prefill attention (+ m, l) and window scores,
                    one selection launch, host block allocation + table upload,
                    one compaction launch;
  decode            500 steps, each: host block preparation, one paged-decode
                    launch over the 32 (request, layer) items;
then the request's blocks are returned to the pool.

Reported: value = prefill+sparsify tokens/s (device time, inputs resident),
decode tokens/s beside it, a roofline object for the dominant kernel
(prefill attention, tensor-bound) and one for the decode kernel (HBM-bound),
the same metrics end to end through host buffers, the CPU oracle timed on a
bounded sample, and the SM clocks sampled during the timed region.

L2: the inputs of one request (1.57 GB of Q/K/V) exceed L2; between decode
steps and between bench steps (outside the timed events) a 512 MB buffer is
written and another 512 MB read, so every decode step starts from a cold L2
with no dirty lines left to write back.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import threading
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "prefill+sparsify tok/s & decode tok/s (1 GB300, 4000/500); % of roofline"
WORKLOAD = "llama3-8b attention shapes, 1 x 4000-token prompt, 500 decode steps, 32 layers"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) of one captured launch, from the ncu captures
# summarised under profiles/, with the algorithmic bytes of that same launch:
# the figure reported is scaled to the launch the bench times (decode length
# grows over the request).  Set an entry to None once its kernel changes.
NCU_TRAFFIC = {
    # the one prefill launch over all 32 layers: the bench's own launch shape
    "prefill_attn": {"bytes": 1694695936 + 1057856512, "alg_bytes": None},
    "paged_decode": {"bytes": 188694528 + 3154432, "alg_bytes": 187432960},
}


# Layers whose prefill-attention and window-score launches get their own
# event pairs (the kernel rooflines): an event between two launches ends the
# overlap of the second one's start with the first one's tail, so the other
# layers run undisturbed inside the timed step.
TIMED_LAYERS = (5, 15, 25)


def max_over_ranks(values, world, dist, device):
    """Per-rank times (ms) -> the largest over all ranks, elementwise (the
    job's time is its slowest replica's).  world == 1: unchanged."""
    if world <= 1:
        return list(values)
    import torch
    tt = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return tt.tolist()


def job_rates(t_pre_ms, t_dec_ms, world, n, steps):
    """Whole-job rates over `world` replicas: prompt tokens/s and decode
    tokens/s from the slowest replica's times."""
    return world * n / (t_pre_ms / 1e3), world * steps / (t_dec_ms / 1e3)


def traffic_for(kernel, alg_bytes=None):
    t = NCU_TRAFFIC.get(kernel)
    if t is None:
        return None
    if t["alg_bytes"] is None or alg_bytes is None:
        return int(t["bytes"])
    return int(round(t["bytes"] * alg_bytes / t["alg_bytes"]))


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return FALLBACK_PEAKS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------
def make_inputs(w, n, steps, device):
    import torch
    from synth import decode_qkv, prefill_qkv
    L = w.n_layers
    q = torch.empty((L, n, w.h_q, w.d), dtype=torch.bfloat16, device=device)
    k = torch.empty((L, n, w.h_kv, w.d), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    dq = torch.empty((steps, L, w.h_q, w.d), dtype=torch.bfloat16, device=device)
    dk = torch.empty((steps, L, w.h_kv, w.d), dtype=torch.bfloat16, device=device)
    dv = torch.empty_like(dk)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    for l in range(L):
        qb, kb, vb = prefill_qkv(w, 0, l, n)
        q[l].copy_(dev(qb))
        k[l].copy_(dev(kb))
        v[l].copy_(dev(vb))
        a, b, c = decode_qkv(w, 0, l, steps)
        dq[:, l].copy_(dev(a))
        dk[:, l].copy_(dev(b))
        dv[:, l].copy_(dev(c))
    return q, k, v, dq, dk, dv


def prefill_flops(w, n):
    """Causal attention work: QK^T and PV over the lower triangle incl. the
    diagonal, all query heads, all layers: 2 * 2 * d * n(n+1)/2 per head."""
    return 2.0 * w.h_q * w.d * n * (n + 1)


def prefill_exps(w, n):
    """Softmax exponentials of the causal prefill of one layer: one per
    (query head, query, key at or before it)."""
    return w.h_q * n * (n + 1) / 2.0


def window_score_flops(w, n, layers):
    """QK^T of the alpha window rows against their visible keys, every query
    head, over `layers` budgeted layers: 2 d (alpha n - alpha (alpha-1) / 2)
    per head."""
    a = min(w.alpha, n)
    return 2.0 * w.h_q * w.d * (a * n - a * (a - 1) / 2.0) * layers


def xu_exp_peak(peaks):
    """Exponentials per second the XU (MUFU) pipes can issue: Blackwell's
    documented rate for ex2 is 16 results per clock per SM, and Blackwell
    Ultra (GB300) doubles the SFU rate of the attention exponential, so 32 per
    clock per SM, times the 152 SMs at the maximum SM clock."""
    return 32.0 * 152 * peaks.get("sm_max_mhz", 2070.0) * 1e6


def prefill_scores_roofline(w, n, flops_launch, k1_avg_ms, k2_ms, peak_t, peak_src, L):
    n_bud = sum(1 for l in range(L) if w.budget(l, n) is not None and w.budget(l, n) < n)
    k2_avg = sum(k2_ms) / max(1, len(k2_ms))
    # one window-score launch covers every budgeted layer when the inputs are
    # resident; the prefill launch covers flops_launch
    layers_per_k1 = flops_launch / prefill_flops(w, n)
    sf = window_score_flops(w, n, n_bud) * layers_per_k1 / L
    ach = (flops_launch + sf) / ((k1_avg_ms + k2_avg) / 1e3) / 1e12
    return {"kernels": "prefill_attn + window_scores", "bound": "tensor",
            "achieved": round(ach, 1), "peak": peak_t, "unit": "TFLOP/s",
            "frac": round(ach / peak_t, 4), "peak_source": f"{peak_src} bf16 burst",
            "flops": flops_launch + sf, "ms": round(k1_avg_ms + k2_avg, 4)}


def decode_bytes(w, lens):
    """Algorithmic bytes of one decode launch: every cached K and V row of
    every item read once (the new row included), q read, out written, the new
    k/v rows written."""
    kv = sum((L + 1) * w.h_kv * w.d * 2 * 2 for L in lens)
    return kv + len(lens) * (w.h_q * w.d * 2 * 2 + w.h_kv * w.d * 2 * 2)


def run_request(eng, dec, w, n, steps, q, k, v, dq, dk, dv, o_buf, ml_buf, flush, rec,
                host=None):
    """One request.  rec: dict collecting event pairs.  host: pinned host
    buffers for the end-to-end variant (inputs copied in, outputs read back
    inside the timed events): the prompt's Q/K/V layer by layer on copy
    streams, each layer's prefill starting once its copies are done; every
    decode step's q/k/v as one packed copy."""
    import torch
    from layer_wise_kv_gb300.pipeline import upload_layers
    L = w.n_layers
    st = torch.cuda.current_stream()
    budgets = [[w.budget(l, n) for l in range(L)]]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st)
    ready = None
    if host is not None:
        ready = upload_layers((host["q"], host["k"], host["v"]), (q, k, v), host["streams"])
    res = eng.prefill_sparsify(list(q), list(k), list(v), [n], budgets, o_buf=o_buf,
                               ml_buf=ml_buf, timing=rec.get("k1"), timing_layers=TIMED_LAYERS,
                               ready=ready)
    if host is not None:
        host["kept"][: res.kept_idx.numel()].copy_(res.kept_idx, non_blocking=True)
    e1.record(st)
    rec["prefill"].append((e0, e1))
    dec.set_stream(0, res.tables[0], res.k_eff[0])
    for t in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        if host is not None:
            host["dqkv_d"][t].copy_(host["dqkv"][t], non_blocking=True)
        out = dec.step(dq[t], dk[t], dv[t], timing=rec.get("dk"))
        if host is not None:
            host["out"][t].copy_(out, non_blocking=True)
        b.record(st)
        rec["decode"].append((a, b))
    torch.cuda.synchronize()
    eng.check_status()
    for s in range(1):
        dec.retire(s)
    return res


def bench_gpu(args):
    import torch
    import torch.distributed as dist
    from synth import llama3_8b
    from layer_wise_kv_gb300 import kvs
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine, Shape, blocks_for

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    kvs.library()

    w = llama3_8b()
    n, steps, L = w.prompt_lens[0], args.decode_steps, w.n_layers
    q, k, v, dq, dk, dv = make_inputs(w, n, steps, dev)
    shape = Shape(w.n_layers, w.h_q, w.h_kv, w.d, w.alpha, w.recent)
    blocks = sum(blocks_for(w.k_eff(l, n) + steps) + 1 for l in range(L))
    eng = Engine(shape, blocks + 64, device=dev)
    o_buf = torch.empty((L, n, w.h_q, w.d), dtype=torch.bfloat16, device=dev)
    ml_buf = (torch.empty((L, w.h_q, n), dtype=torch.float32, device=dev),
              torch.empty((L, w.h_q, n), dtype=torch.float32, device=dev))
    scrub = torch.ones(128 << 20, dtype=torch.int32, device=dev)   # 512 MB
    scrub_r = torch.ones(128 << 20, dtype=torch.int32, device=dev)
    dec = DecodeBatch(eng, 1, n + steps)

    def flush():
        # write 512 MB (> L2) so the next step starts cold, then read another
        # 512 MB so the dirty lines are written back before, not during, the
        # timed kernels
        scrub.fill_(1)
        scrub_r.sum(dtype=torch.int32)

    def new_rec(k1=True):
        return {"prefill": [], "decode": [], "k1": {"attn": [], "scores": []} if k1 else None,
                "dk": [] if k1 else None}

    # warm-up
    for _ in range(args.warmup):
        run_request(eng, dec, w, n, steps, q, k, v, dq, dk, dv, o_buf, ml_buf, flush,
                    new_rec(False))
    flush()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    # no Python garbage collection inside the timed region: a collection
    # pauses the host thread that enqueues the work (tens of ms after the
    # warm-up's allocations) and the GPU idles meanwhile
    gc.collect()
    gc.disable()
    rec = new_rec()
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        flush()
        run_request(eng, dec, w, n, steps, q, k, v, dq, dk, dv, o_buf, ml_buf, flush, rec)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    gc.enable()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()

    pre_ms = [a.elapsed_time(b) for a, b in rec["prefill"]]
    dec_ms = [a.elapsed_time(b) for a, b in rec["decode"]]
    k1_ms = [a.elapsed_time(b) for a, b in rec["k1"]["attn"]]
    k2_ms = [a.elapsed_time(b) for a, b in rec["k1"]["scores"]]
    t_pre = sum(pre_ms) / args.steps            # ms per request
    t_dec = sum(dec_ms) / args.steps
    t_pre, t_dec = max_over_ranks([t_pre, t_dec], world, dist, dev)
    prefill_tok_s, decode_tok_s = job_rates(t_pre, t_dec, world, n, steps)

    peaks, peak_src = read_peaks()
    k1_avg = sum(k1_ms) / len(k1_ms)
    # layers per timed prefill launch (all 32 when the layers go in one launch)
    k1_layers = rec["k1"].get("attn_layers") or [1] * len(k1_ms)
    flops_launch = prefill_flops(w, n) * (sum(k1_layers) / len(k1_layers))
    tflops = flops_launch / (k1_avg / 1e3) / 1e12
    exps_launch = prefill_exps(w, n) * (sum(k1_layers) / len(k1_layers))
    exp_rate = exps_launch / (k1_avg / 1e3)
    # the prefill launch runs a few ms at the maximum clock inside a step, not
    # a seconds-long power-capped loop: the burst figure is its peak
    peak_t = peaks["bf16_tflops"]
    dk_ms = [a.elapsed_time(b) for a, b in rec["dk"]]
    dec_avg = sum(dk_ms) / len(dk_ms)            # the decode kernel alone
    lens = [w.k_eff(l, n) + steps // 2 for l in range(L)]   # mean length over the request
    gbs = decode_bytes(w, lens) / (dec_avg / 1e3) / 1e9

    out = {
        "metric": METRIC,
        "value": round(prefill_tok_s, 1),
        "unit": "tok/s",
        "decode": {"value": round(decode_tok_s, 1), "unit": "tok/s",
                   "ms_per_token": round(t_dec / steps, 4)},
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_pre + t_dec, 3),
        "ms_prefill_sparsify": round(t_pre, 3),
        "ms_decode_500": round(t_dec, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V with sink tokens; no weights)",
        "config": {"workload": WORKLOAD, "prompt": n, "decode_steps": steps, "layers": L,
                   "h_q": w.h_q, "h_kv": w.h_kv, "d": w.d, "alpha": w.alpha,
                   "recent": w.recent, "budgets": "layers 0-2 full, 2048-64*(l-3)",
                   "l2": "inputs 1.57 GB > L2; 512 MB written then 512 MB read between decode steps (L2 flush)",
                   "parallelism": f"replicas x{world}"},
        # the dominant kernel of a step by device time: paged decode (about
        # 87 % of a step's device time)
        "roofline": {"kernel": "paged_decode (+ split merge, one call)", "bound": "hbm",
                     "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / peaks["hbm_gbs"], 4),
                     "traffic": traffic_for("paged_decode", decode_bytes(w, lens)),
                     "peak_source": f"{peak_src} copy bandwidth",
                     "per_launch_ms": round(dec_avg, 4),
                     "bytes_per_launch": decode_bytes(w, lens),
                     "step_ms": round(sum(dec_ms) / len(dec_ms), 4)},
        "roofline_prefill": {"kernel": "prefill_attn (tcgen05)", "bound": "tensor",
                             "achieved": round(tflops, 1), "peak": peak_t, "unit": "TFLOP/s",
                             "frac": round(tflops / peak_t, 4),
                             "traffic": traffic_for("prefill_attn"),
                             "peak_source": f"{peak_src} bf16 burst",
                             "per_launch_ms": round(k1_avg, 4), "flops_per_launch": flops_launch,
                             # the softmax's exponentials (every one an ex2 on the XU pipe)
                             # against the XU peak derived in xu_exp_peak()
                             "exp_per_launch": exps_launch,
                             "exp_per_s": round(exp_rate, -6),
                             "exp_peak_per_s": round(xu_exp_peak(peaks), -6),
                             "exp_frac": round(exp_rate / xu_exp_peak(peaks), 4)},
        # prefill attention and window scores together, as one tensor-bound
        # stage: both launches' flops over both launches' event time
        "roofline_prefill_scores": prefill_scores_roofline(w, n, flops_launch, k1_avg, k2_ms,
                                                           peak_t, peak_src, L),
        # one window-score launch per request covers the budgeted layers
        "scores_ms_per_launch": round(sum(k2_ms) / max(1, len(k2_ms)), 4),
        "scores_layers_per_launch": sum(1 for l in range(L) if w.budget(l, n) is not None
                                        and w.budget(l, n) < n),
        # per timed request: the prefill launch(es), the window-score launch(es)
        # (one event pair around each), selection, compaction, and each decode
        # step's decode + merge
        "gpu_launches": args.steps * ((1 if all(x == L for x in k1_layers) else L)
                                      + len(k2_ms) // max(1, args.steps) + 2 + 2 * steps),
        "clocks": clk,
        "wall_s": round(t_wall, 2),
    }
    if args.decode_wall:
        out["decode_wall"] = bench_decode_wall(args, eng, dec, w, n, steps, q, k, v, dq, dk, dv,
                                               o_buf, ml_buf, world, dist)
    if args.decode_evicting:
        out["decode_evicting"] = bench_decode_evicting(args, eng, w, n, steps, q, k, v, dq, dk,
                                                       dv, o_buf, ml_buf, flush, world, dist)
    if args.decode_fp8:
        out["decode_fp8"] = bench_decode_fp8(args, shape, blocks + 64, w, n, steps, q, k, v, dq,
                                             dk, dv, o_buf, ml_buf, flush, world, dist)
    if args.decode_per_layer:
        out["decode_per_layer"] = bench_decode_per_layer(args, eng, w, n, steps, q, k, v, dq, dk,
                                                         dv, o_buf, ml_buf, flush, world, dist)
    if args.prefill_per_layer:
        out["prefill_per_layer"] = bench_prefill_per_layer(args, eng, dec, w, n, q, k, v, ml_buf,
                                                           flush, world, dist)
    if args.e2e:
        out["e2e"] = bench_e2e(args, eng, dec, w, n, steps, q, k, v, dq, dk, dv, o_buf, ml_buf,
                               flush, world, dist)
    if args.c2:
        out["c2_serving"] = bench_c2_serving(args, w, q, k, v, dq, dk, dv, dev, world, dist)
    if args.c3:
        del o_buf, ml_buf
        torch.cuda.empty_cache()
        out["c3_long_context"] = bench_c3_long_context(args, dev, world, dist)
    if args.c4:
        out["c4_shared_prefix"] = bench_c4_shared_prefix(args, dev, world, dist)
    if rank == 0 and args.cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args)
        out["cpu_baseline"]["parallel"] = cpu_baseline_parallel(args)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def bench_decode_wall(args, eng, dec, w, n, steps, q, k, v, dq, dk, dv, o_buf, ml_buf, world,
                      dist):
    """Decode as a serving loop runs it: the request's steps back to back,
    each one native call (host allocator preparation, uploads, decode and
    merge), timed by the host clock from the first step's call to the last
    step's completion, so host work counts.  No L2 flush between steps: each
    step reads about 220 MB of K/V, more than L2 holds.  Median of three
    requests (after one untimed)."""
    import torch
    L = w.n_layers
    budgets = [[w.budget(l, n) for l in range(L)]]
    rates = []
    for rep in range(4):
        res = eng.prefill_sparsify(list(q), list(k), list(v), [n], budgets, o_buf=o_buf,
                                   ml_buf=ml_buf)
        dec.set_stream(0, res.tables[0], res.k_eff[0])
        # each step's inputs as ready tensors, the way a model hands them over
        step_in = list(zip(dq.unbind(0), dk.unbind(0), dv.unbind(0)))
        torch.cuda.synchronize()
        gc.collect()
        gc.disable()
        t0 = time.perf_counter()
        for qt, kt, vt in step_in:
            dec.step(qt, kt, vt)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        gc.enable()
        eng.check_status()
        dec.retire(0)
        if rep > 0:
            rates.append(dt)
    dt = sorted(rates)[len(rates) // 2]
    (dt,) = max_over_ranks([dt * 1e3], world, dist, q.device)
    return {"value": round(world * steps / (dt / 1e3), 1), "unit": "tok/s",
            "ms_per_token": round(dt / steps, 4),
            "what": "500 back-to-back native decode steps (host allocator + uploads + decode + "
                    "merge), host wall clock, no L2 flush (220 MB per step > L2)"}


def bench_decode_evicting(args, eng, w, n, steps, q, k, v, dq, dk, dv, o_buf, ml_buf, flush,
                          world, dist):
    """Decode with decode-time replacement in the budgeted layers (3-31 keep
    exactly k_l slots: each step's token replaces the lowest-scoring one
    outside the recent window), the full-cache layers 0-2 growing as usual:
    the request's 500 steps with the same L2 flush and per-step events as the
    headline decode.  Bytes per step: the K/V rows every step reads (full
    layers at the mean length, budgeted layers at k_l) plus the budgeted
    layers' logits written by the decode launch and read by the score update.
    Over FP8 pools (eng.kv_fp8) a row is its d codes and 4-byte scale."""
    import torch
    from layer_wise_kv_gb300.pipeline import DecodeBatch, EvictingDecode
    L = w.n_layers
    budgets = [[w.budget(l, n) for l in range(L)]]
    full = [l for l in range(L) if w.budget(l, n) is None or w.budget(l, n) >= n]
    bud = [l for l in range(L) if l not in full]
    res = eng.prefill_sparsify(list(q), list(k), list(v), [n], budgets, o_buf=o_buf, ml_buf=ml_buf)
    dec_f = DecodeBatch(eng, 1, n + steps, n_layers=len(full))
    dec_f.set_stream(0, [res.tables[0][l] for l in full], [res.k_eff[0][l] for l in full])
    ev = EvictingDecode(eng, res, 0, 0, n, bud)
    fq, fk, fv = (x[:, full].contiguous() for x in (dq, dk, dv))
    bq, bk, bv = (x[:, bud].contiguous() for x in (dq, dk, dv))
    torch.cuda.synchronize()
    pairs = []
    gc.collect()
    gc.disable()
    for t in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        dec_f.step(fq[t], fk[t], fv[t])
        ev.step(bq[t], bk[t], bv[t])
        b.record()
        pairs.append((a, b))
    torch.cuda.synchronize()
    gc.enable()
    eng.check_status()
    dec_f.retire(0)
    ev.release()
    t_ms = sum(a.elapsed_time(b) for a, b in pairs)
    (t_ms,) = max_over_ranks([t_ms], world, dist, q.device)
    row = w.h_kv * (w.d + 4) if eng.kv_fp8 else w.h_kv * w.d * 2
    kv_full = sum((w.k_eff(l, n) + steps // 2 + 1) * row * 2 for l in full)
    kv_bud = sum(w.k_eff(l, n) * row * 2 for l in bud)
    # the decode launch writes the budgeted slots' logits (fp32, per query
    # head) and the score update reads them back
    logit_bytes = sum(w.k_eff(l, n) * w.h_q * 4 * 2 for l in bud)
    bytes_step = kv_full + kv_bud + logit_bytes
    per = t_ms / steps
    peaks, _ = read_peaks()
    return {"value": round(world * steps / (t_ms / 1e3), 1), "unit": "tok/s",
            "ms_per_token": round(per, 4), "bytes_per_step": int(bytes_step),
            "achieved_gbs": round(bytes_step / (per / 1e3) / 1e9, 1),
            "frac_of_hbm": round(bytes_step / (per / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
            "what": "layers 3-31 replace their lowest-scoring token each step (k_l slots kept), "
                    "layers 0-2 grow; events per step, L2 flushed before each"}


def bench_decode_fp8(args, shape, num_blocks, w, n, steps, q, k, v, dq, dk, dv, o_buf, ml_buf,
                     flush, world, dist):
    """The headline request's decode over FP8 pools (e4m3 codes, per-row fp32
    scales): the prefill compacts into them, then 500 steps, each the
    allocator's preparation, the table-patch upload and one FP8 decode
    launch over the 32 layers, with the same L2 flush and per-step events as
    the headline decode; kernel events around each decode launch give the
    roofline.  Bytes per decode launch: every cached row's d codes and 4-byte
    scale, K and V, plus q, out and the new rows."""
    import torch
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine
    L = w.n_layers
    budgets = [[w.budget(l, n) for l in range(L)]]
    eng8 = Engine(shape, num_blocks, device=q.device, kv_dtype="fp8")
    dec8 = DecodeBatch(eng8, 1, n + steps)
    res = eng8.prefill_sparsify(list(q), list(k), list(v), [n], budgets, o_buf=o_buf,
                                ml_buf=ml_buf)
    dec8.set_stream(0, res.tables[0], res.k_eff[0])
    torch.cuda.synchronize()
    pairs, kern = [], []
    gc.collect()
    gc.disable()
    for t in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        dec8.step(dq[t], dk[t], dv[t], timing=kern)
        b.record()
        pairs.append((a, b))
    torch.cuda.synchronize()
    gc.enable()
    eng8.check_status()
    dec8.retire(0)
    # the same request with decode-time replacement over the FP8 pools
    evicting = bench_decode_evicting(args, eng8, w, n, steps, q, k, v, dq, dk, dv, o_buf, ml_buf,
                                     flush, world, dist)
    evicting["what"] = ("over the FP8 pools: " + evicting["what"] + "; the new row is "
                        "quantised into the replaced slot")
    t_ms = sum(a.elapsed_time(b) for a, b in pairs)
    k_ms = sum(a.elapsed_time(b) for a, b in kern)
    t_ms, k_ms = max_over_ranks([t_ms, k_ms], world, dist, q.device)
    row = w.h_kv * (w.d + 4)
    lens = [w.k_eff(l, n) for l in range(L)]
    per_launch = []
    for t in range(steps):
        kv = sum((Lq + t + 1) * row * 2 for Lq in lens)
        per_launch.append(kv + L * (w.h_q * w.d * 2 * 2 + w.h_kv * w.d * 2 * 2))
    alg = sum(per_launch) / steps
    per_k = k_ms / steps
    peaks, _ = read_peaks()
    ach = alg / (per_k / 1e3) / 1e9
    del dec8, eng8
    return {"value": round(world * steps / (t_ms / 1e3), 1), "unit": "tok/s",
            "ms_per_token": round(t_ms / steps, 4), "kernel_ms": round(per_k, 4),
            "bytes_per_launch": int(alg), "achieved_gbs": round(ach, 1),
            "frac_of_hbm": round(ach / peaks["hbm_gbs"], 4),
            "what": "decode over e4m3 pools with per-row scales (codes + scales read), "
                    "eager steps with allocator preparation, events per step, L2 flushed "
                    "before each",
            "evicting": evicting}


def _step_bytes(w, lens_h):
    """Algorithmic bytes of one decode step over items whose lengths before
    the step are lens_h (each appends one token)."""
    return decode_bytes(w, [int(x) for x in lens_h])


def bench_decode_per_layer(args, eng, w, n, steps, q, k, v, dq, dk, dv, o_buf, ml_buf, flush,
                           world, dist):
    """The headline request's decode in model order: each step is one host
    preparation and then one decode launch per layer (32 launches of one item,
    each with its merge), as a model issues them (layer l + 1's query needs
    layer l's output), replayed from a CUDA graph per step; events per step,
    L2 flushed before each, bytes as the headline decode."""
    import torch
    from layer_wise_kv_gb300.pipeline import DecodeBatch
    L = w.n_layers
    budgets = [[w.budget(l, n) for l in range(L)]]
    decl = DecodeBatch(eng, 1, n + steps, layer_order=True)
    res = eng.prefill_sparsify(list(q), list(k), list(v), [n], budgets, o_buf=o_buf,
                               ml_buf=ml_buf)
    decl.set_stream(0, res.tables[0], res.k_eff[0])
    decl.capture_graphs()
    torch.cuda.synchronize()
    pairs, nbytes = [], 0
    gc.collect()
    gc.disable()
    for t in range(steps):
        flush()
        nbytes += _step_bytes(w, decl.lens_h)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        decl.step(dq[t], dk[t], dv[t])
        b.record()
        pairs.append((a, b))
    torch.cuda.synchronize()
    gc.enable()
    eng.check_status()
    decl.retire(0)
    del decl
    t_ms = sum(a.elapsed_time(b) for a, b in pairs)
    (t_ms,) = max_over_ranks([t_ms], world, dist, q.device)
    peaks, src = read_peaks()
    ach = nbytes / (t_ms / 1e3) / 1e9
    return {"value": round(world * steps / (t_ms / 1e3), 1), "unit": "tok/s",
            "ms_per_token": round(t_ms / steps, 4), "launches_per_step": 2 * L,
            "bytes_per_step": int(nbytes / steps), "achieved_gbs": round(ach, 1),
            "frac_of_hbm": round(ach / peaks["hbm_gbs"], 4),
            "what": "one decode launch (+ merge) per layer per step, 32 x 1 item, the step "
                    "replayed from a CUDA graph after the host allocator's preparation; events "
                    "per step, L2 flushed before each"}


def bench_prefill_per_layer(args, eng, dec, w, n, q, k, v, ml_buf, flush, world, dist):
    """The request's prefill+sparsify with one prefill-attention launch per
    layer, the order a model issues them (layer l + 1's Q, K and V need layer
    l's output): every layer overwrites one [n][h_q][d] output buffer; the
    window scores, selection and compaction follow as in the headline.  Events
    around the call (L2 flushed before each); the attention roofline from
    event pairs around the launches of layers 5, 15 and 25."""
    import torch
    L = w.n_layers
    budgets = [[w.budget(l, n) for l in range(L)]]
    o_layer = torch.empty((n, w.h_q, w.d), dtype=torch.bfloat16, device=q.device)
    totals, k1 = [], {}
    for rep in range(1 + max(1, args.steps)):
        flush()
        tm = {} if rep == 0 else k1
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        res = eng.prefill_sparsify(list(q), list(k), list(v), [n], budgets, o_buf=o_layer,
                                   ml_buf=ml_buf, timing=tm, timing_layers=TIMED_LAYERS)
        e1.record()
        torch.cuda.synchronize()
        eng.check_status()
        if rep > 0:
            totals.append(e0.elapsed_time(e1))
        dec.set_stream(0, res.tables[0], res.k_eff[0])
        dec.retire(0)
    attn = [a.elapsed_time(b) for a, b in k1.get("attn", [])]
    t_ms = sum(totals) / len(totals)
    a_ms = sum(attn) / max(1, len(attn))
    t_ms, a_ms = max_over_ranks([t_ms, a_ms], world, dist, q.device)
    peaks, peak_src = read_peaks()
    tf = prefill_flops(w, n) / (a_ms / 1e3) / 1e12
    return {"value": round(world * n / (t_ms / 1e3), 1), "unit": "tok/s",
            "ms_prefill_sparsify": round(t_ms, 3),
            "roofline_attn_layer": {"achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
                                    "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                                    "per_launch_ms": round(a_ms, 4),
                                    "flops_per_launch": prefill_flops(w, n),
                                    "peak_source": f"{peak_src} bf16 burst"},
            "what": ("prefill+sparsify with 32 prefill-attention launches (one per layer, each "
                     "overwriting one output buffer), then one window-score launch, selection "
                     "and compaction; events around the call, L2 flushed before each")}


def device_prompts(w, lens, layers, seed, dev):
    """Seeded synthetic prompt Q/K/V generated on the device (torch's Philox
    generator), packed [L][T][h][d] bf16: N(0,1) with the sink construction of
    the workloads (keys at positions 0 and 37 of each sequence + 6u, every
    query + 0.5u, u the workload's seeded unit vector), for timing runs whose
    inputs are too large to draw on the host in reasonable time."""
    import torch
    from synth import sink_direction
    from synth.workloads import SINK_KEY_GAIN, SINK_POSITIONS, SINK_QUERY_GAIN
    T = int(sum(lens))
    u = torch.from_numpy(sink_direction(w)).to(dev)
    g = torch.Generator(device=dev)
    out = [torch.empty((layers, T, h, w.d), dtype=torch.bfloat16, device=dev)
           for h in (w.h_q, w.h_kv, w.h_kv)]
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(int)
    for l in range(layers):
        for kind, (buf, h) in enumerate(zip(out, (w.h_q, w.h_kv, w.h_kv))):
            g.manual_seed(seed * 1000003 + l * 4 + kind)
            x = torch.randn((T, h, w.d), generator=g, device=dev, dtype=torch.float32)
            if kind == 0:
                x += SINK_QUERY_GAIN * u
            elif kind == 1:
                for s0, nb in zip(starts, lens):
                    for p in SINK_POSITIONS:
                        if p < nb:
                            x[s0 + p] += SINK_KEY_GAIN * u
            buf[l].copy_(x)
            del x
    return out


def bench_c2_serving(args, w1, q, k, v, dq, dk, dv, dev, world, dist):
    """Continuous batching at the pages' serving point: 20 live 4000-token
    sequences, 40 in all, output lengths drawn in [400, 600]; a finished
    sequence's blocks go back to the free list (a seeded shuffle at the start)
    and its slot is refilled by the next sequence at once (one prefill of one
    prompt); the first 20 are admitted with one packed prefill of 20 prompts.
    Every prompt is the headline request's 4000-token prompt (resident) and
    every step's q/k/v the headline request's decode inputs for that layer,
    replicated over the streams: the shapes and lengths are the workload's,
    the values do not change the work.  Two passes: one decode launch per step
    over all 640 items (stream-major), and model order (one launch per layer
    over its 20 items, each step replayed from a CUDA graph).  Events around
    every prefill call and every decode step; no L2 flush (a step reads about
    4.4 GB).  Decode bytes: every live item's cached rows (+ the new one),
    q, out and new rows, from the host mirror of the lengths."""
    import torch
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine, Shape, blocks_for
    from synth import continuous_batching, shuffled_block_order
    wc = continuous_batching()
    conc, prompts, outs = wc.concurrency, [int(x) for x in wc.prompt_lens], \
        [int(x) for x in wc.out_lens]
    n = prompts[0]
    assert all(p == n for p in prompts) and n == q.shape[1]
    L, steps_in = wc.n_layers, dq.shape[0]
    shape = Shape(L, wc.h_q, wc.h_kv, wc.d, wc.alpha, wc.recent)
    per_seq = sum(blocks_for(wc.k_eff(l, n) + max(outs) + 1) for l in range(L))
    N = conc * per_seq + 64
    budgets1 = [[wc.budget(l, n) for l in range(L)]]
    q20, k20, v20 = (x.repeat(1, conc, 1, 1) for x in (q, k, v))
    o20 = torch.empty((L, conc * n, wc.h_q, wc.d), dtype=torch.bfloat16, device=dev)
    ml20 = (torch.empty((L, wc.h_q, conc * n), dtype=torch.float32, device=dev),
            torch.empty((L, wc.h_q, conc * n), dtype=torch.float32, device=dev))
    o1 = torch.empty((L, n, wc.h_q, wc.d), dtype=torch.bfloat16, device=dev)
    ml1 = (torch.empty((L, wc.h_q, n), dtype=torch.float32, device=dev),
           torch.empty((L, wc.h_q, n), dtype=torch.float32, device=dev))
    # decode inputs per step for every item: [steps][S*L] stream-major and
    # [steps][L*S] layer-major
    sm = [x[:, None].expand(steps_in, conc, L, *x.shape[2:]).reshape(steps_in, conc * L,
                                                                     *x.shape[2:]).contiguous()
          for x in (dq, dk, dv)]
    lm = [x[:, :, None].expand(steps_in, L, conc, *x.shape[2:]).reshape(steps_in, conc * L,
                                                                       *x.shape[2:]).contiguous()
          for x in (dq, dk, dv)]
    peaks, src = read_peaks()
    result = {}
    for mode in ("batched", "layer_order"):
        eng = Engine(shape, N, device=dev, initial_free=shuffled_block_order(N, 1))
        dec = DecodeBatch(eng, conc, n + max(outs) + 1, layer_order=(mode == "layer_order"))
        inputs = lm if mode == "layer_order" else sm
        pre, stp, live = [], [], {}
        nbytes = tokens = 0

        def timed(fn):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            r = fn()
            b.record()
            return r, (a, b)

        torch.cuda.synchronize()
        gc.collect()
        gc.disable()
        res, ev = timed(lambda: eng.prefill_sparsify(list(q20), list(k20), list(v20),
                                                     [n] * conc, budgets1 * conc, o_buf=o20,
                                                     ml_buf=ml20))
        pre.append(ev)
        for s in range(conc):
            dec.set_stream(s, res.tables[s], res.k_eff[s])
            live[s] = [s, 0]
        if mode == "layer_order":
            dec.capture_graphs()
        nxt, t = conc, 0
        while True:
            nbytes += _step_bytes(wc, dec.lens_h)
            _, ev = timed(lambda: dec.step(inputs[0][t % steps_in], inputs[1][t % steps_in],
                                           inputs[2][t % steps_in]))
            stp.append(ev)
            tokens += conc
            t += 1
            done = False
            for s in range(conc):
                live[s][1] += 1
                if live[s][1] >= outs[live[s][0]]:
                    dec.retire(s)
                    if nxt >= len(prompts):
                        done = True
                        continue
                    r1, ev = timed(lambda: eng.prefill_sparsify(list(q), list(k), list(v), [n],
                                                                budgets1, o_buf=o1, ml_buf=ml1))
                    pre.append(ev)
                    dec.set_stream(s, r1.tables[0], r1.k_eff[0])
                    live[s] = [nxt, 0]
                    nxt += 1
            if done:
                break
        torch.cuda.synchronize()
        gc.enable()
        eng.check_status()
        t_pre = sum(a.elapsed_time(b) for a, b in pre)
        t_dec = sum(a.elapsed_time(b) for a, b in stp)
        t_pre, t_dec = max_over_ranks([t_pre, t_dec], world, dist, dev)
        ach = nbytes / (t_dec / 1e3) / 1e9
        entry = {"decode_tok_s": round(world * tokens / (t_dec / 1e3), 1),
                 "decode_steps": t, "ms_per_step": round(t_dec / t, 4),
                 "bytes_per_step": int(nbytes / t), "achieved_gbs": round(ach, 1),
                 "frac_of_hbm": round(ach / peaks["hbm_gbs"], 4),
                 "launches_per_step": 2 * (L if mode == "layer_order" else 1)}
        if mode == "batched":
            entry = {"prefill_sparsify_tok_s": round(world * len(prompts) * n / (t_pre / 1e3), 1),
                     "prefill_calls": len(pre), **entry}
        result[mode] = entry
        for s in range(conc):
            if dec.lens_h[dec._item(s, 0)] > 0:
                dec.retire(s)
        del dec, eng
    del q20, k20, v20, o20, ml20, sm, lm
    torch.cuda.empty_cache()
    result["what"] = ("20 live of 40 sequences, 4000-token prompts, outputs U[400,600], seeded "
                      "shuffled free list; prefill+sparsify = 40 prompts over all prefill calls; "
                      "decode 'batched' = one launch over all 640 items per step, 'layer_order' "
                      "= 32 launches of 20 items per step from a CUDA graph; no L2 flush "
                      "(4.4 GB per step)")
    result["peak_source"] = f"{src} copy bandwidth"
    return result


def bench_c3_long_context(args, dev, world, dist):
    """Long context at >10x compression: one batch of four prompts of 7000,
    12000, 20000 and 30000 tokens (Llama-3-8B head shapes; layers 0-2 full,
    layers 3-31 keep floor(n/12) incl. the 32 most recent), prefill+sparsify
    as one call (one prefill launch over all layers and sequences), then 64
    decode steps over the 128 items.  Inputs drawn on the device (seeded) with
    the workloads' distribution and sinks.  Events around the call and around
    the prefill-attention launch (its roofline at these lengths) and each
    decode step; no L2 flush (a step reads about 1.5 GB)."""
    import torch
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine, Shape, blocks_for
    from synth import long_context
    wl = long_context()
    lens = [int(x) for x in wl.prompt_lens]
    L, steps, T = wl.n_layers, wl.decode_steps, sum(lens)
    shape = Shape(L, wl.h_q, wl.h_kv, wl.d, wl.alpha, wl.recent)
    q, k, v = device_prompts(wl, lens, L, 3, dev)
    budgets = [[wl.budget(l, nb) for l in range(L)] for nb in lens]
    N = sum(blocks_for(wl.k_eff(l, nb) + steps + 1) for nb in lens for l in range(L)) + 64
    eng = Engine(shape, N, device=dev)
    o_buf = torch.empty((L, T, wl.h_q, wl.d), dtype=torch.bfloat16, device=dev)
    ml_buf = (torch.empty((L, wl.h_q, T), dtype=torch.float32, device=dev),
              torch.empty((L, wl.h_q, T), dtype=torch.float32, device=dev))
    g = torch.Generator(device=dev)
    g.manual_seed(77)
    dqs = [torch.randn((steps, len(lens) * L, h, wl.d), generator=g, device=dev).bfloat16()
           for h in (wl.h_q, wl.h_kv, wl.h_kv)]
    peaks, src = read_peaks()
    pre, k1, stp, nbytes = [], [], [], 0
    reps = 2
    for rep in range(reps + 1):                      # the first pass is a warm-up
        torch.cuda.synchronize()
        tm = {"attn": [], "scores": []}
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        res = eng.prefill_sparsify(list(q), list(k), list(v), lens, budgets, o_buf=o_buf,
                                   ml_buf=ml_buf, timing=tm)
        b.record()
        if rep > 0:
            pre.append((a, b))
            k1 += tm["attn"]
        dec = DecodeBatch(eng, len(lens), max(lens) + steps + 1)
        for s in range(len(lens)):
            dec.set_stream(s, res.tables[s], res.k_eff[s])
        for t in range(steps):
            if rep > 0:
                nbytes += _step_bytes(wl, dec.lens_h)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            dec.step(dqs[0][t], dqs[1][t], dqs[2][t])
            b.record()
            if rep > 0:
                stp.append((a, b))
        torch.cuda.synchronize()
        eng.check_status()
        for s in range(len(lens)):
            dec.retire(s)
        del dec
    t_pre = sum(a.elapsed_time(b) for a, b in pre) / reps
    t_k1 = sum(a.elapsed_time(b) for a, b in k1) / reps
    t_dec = sum(a.elapsed_time(b) for a, b in stp) / reps
    t_pre, t_k1, t_dec = max_over_ranks([t_pre, t_k1, t_dec], world, dist, dev)
    flops = sum(prefill_flops(wl, nb) for nb in lens) * L
    tf = flops / (t_k1 / 1e3) / 1e12
    ach = nbytes / reps / (t_dec / 1e3) / 1e9
    del q, k, v, o_buf, ml_buf, dqs, eng
    torch.cuda.empty_cache()
    return {"prefill_sparsify_tok_s": round(world * T / (t_pre / 1e3), 1),
            "ms_prefill_sparsify": round(t_pre, 3),
            "roofline_prefill": {"achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
                                 "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                                 "flops_per_launch": flops, "per_launch_ms": round(t_k1, 4),
                                 "peak_source": f"{src} bf16 burst"},
            "decode_tok_s": round(world * len(lens) * steps / (t_dec / 1e3), 1),
            "decode_ms_per_step": round(t_dec / steps, 4),
            "decode_bytes_per_step": int(nbytes / reps / steps),
            "decode_frac_of_hbm": round(ach / peaks["hbm_gbs"], 4),
            "what": "batch of 4 prompts (7000/12000/20000/30000), layers 3-31 keep n/12, one "
                    "prefill+sparsify call, 64 decode steps (one launch over 128 items each); "
                    "inputs drawn on the device; no L2 flush (1.5 GB per step)"}


def bench_c4_shared_prefix(args, dev, world, dist):
    """Shared prefix: 16 prompts of 512 .. 16384 tokens (seeded), one
    prefill+sparsify call over all 32 layers, then each prompt decoded as
    three parallel samples that share its blocks through reference counts; a
    sample's first write into a partially filled last block copies it
    (copy-on-write).  256 decode steps over the 16 x 3 x 32 items.  Inputs
    drawn on the device; events around the call and each decode step (one
    warm-up pass first); no L2 flush (a step reads about 11 GB)."""
    import torch
    from layer_wise_kv_gb300.pipeline import DecodeBatch, Engine, Shape, blocks_for
    from synth import shared_prefix
    wl = shared_prefix()
    lens = [int(x) for x in wl.prompt_lens]
    P, S = len(lens), wl.samples
    L, steps, T = wl.n_layers, wl.decode_steps, sum(lens)
    shape = Shape(L, wl.h_q, wl.h_kv, wl.d, wl.alpha, wl.recent)
    q, k, v = device_prompts(wl, lens, L, 4, dev)
    budgets = [[wl.budget(l, nb) for l in range(L)] for nb in lens]
    base = sum(blocks_for(wl.k_eff(l, nb)) for nb in lens for l in range(L))
    growth = sum(blocks_for(wl.k_eff(l, nb) + steps) - blocks_for(wl.k_eff(l, nb)) + 1
                 for nb in lens for l in range(L))
    N = base + S * growth + 64
    eng = Engine(shape, N, device=dev)
    o_buf = torch.empty((L, T, wl.h_q, wl.d), dtype=torch.bfloat16, device=dev)
    ml_buf = (torch.empty((L, wl.h_q, T), dtype=torch.float32, device=dev),
              torch.empty((L, wl.h_q, T), dtype=torch.float32, device=dev))
    g = torch.Generator(device=dev)
    g.manual_seed(78)
    dqs = [torch.randn((steps, P * S * L, h, wl.d), generator=g, device=dev).bfloat16()
           for h in (wl.h_q, wl.h_kv, wl.h_kv)]
    peaks, _ = read_peaks()
    pre, stp, nbytes, ubytes = [], [], 0, 0
    row = wl.h_kv * wl.d * 2 * 2                     # one token's K and V row, one head set
    for rep in range(2):                             # the first pass is a warm-up
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        res = eng.prefill_sparsify(list(q), list(k), list(v), lens, budgets, o_buf=o_buf,
                                   ml_buf=ml_buf)
        b.record()
        if rep > 0:
            pre.append((a, b))
        # layer-major numbering in one launch: a prompt's three samples sit
        # side by side in the split, so their reads of shared blocks meet in L2
        dec = DecodeBatch(eng, P * S, max(lens) + steps + 1, interleave=True)
        for pi in range(P):
            dec.set_stream(pi * S, res.tables[pi], res.k_eff[pi])
            for si in range(1, S):
                for t in res.tables[pi]:
                    for blk in t:
                        eng.alloc.incref(blk)
                dec.set_stream(pi * S + si, res.tables[pi], res.k_eff[pi])
        # the full blocks of a prompt's kept rows stay shared by its samples;
        # each sample owns the rest (its copy of the partial last block and
        # every appended row)
        shared = [[(ke // 16) * 16 for ke in res.k_eff[pi]] for pi in range(P)]
        for t in range(steps):
            if rep > 0:
                nbytes += _step_bytes(wl, dec.lens_h)
                ubytes += sum(sh + S * (ke - sh + t + 1)
                              for pi in range(P)
                              for sh, ke in zip(shared[pi], res.k_eff[pi])) * row
                ubytes += P * S * L * (wl.h_q * wl.d * 2 * 2 + row)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            dec.step(dqs[0][t], dqs[1][t], dqs[2][t])
            b.record()
            if rep > 0:
                stp.append((a, b))
        torch.cuda.synchronize()
        eng.check_status()
        for si in range(P * S):
            dec.retire(si)
        del dec
    t_pre = sum(a.elapsed_time(b) for a, b in pre)
    t_dec = sum(a.elapsed_time(b) for a, b in stp)
    t_pre, t_dec = max_over_ranks([t_pre, t_dec], world, dist, dev)
    ach = ubytes / (t_dec / 1e3) / 1e9
    del q, k, v, o_buf, ml_buf, dqs, eng
    torch.cuda.empty_cache()
    return {"prefill_sparsify_tok_s": round(world * T / (t_pre / 1e3), 1),
            "ms_prefill_sparsify": round(t_pre, 3),
            "decode_tok_s": round(world * P * S * steps / (t_dec / 1e3), 1),
            "decode_ms_per_step": round(t_dec / steps, 4),
            # every sample's reads (the shared blocks once per sample, two of
            # three then come from L2) and the bytes DRAM must supply (the
            # shared blocks once per step): the roofline is on the second
            "decode_read_bytes_per_step": int(nbytes / steps),
            "decode_read_gbs": round(nbytes / (t_dec / 1e3) / 1e9, 1),
            "decode_bytes_per_step": int(ubytes / steps),
            "decode_frac_of_hbm": round(ach / peaks["hbm_gbs"], 4),
            "what": (f"16 prompts ({T} tokens, 512..16384 each), one prefill+sparsify call, "
                     "then three samples per prompt sharing its blocks (reference counts, "
                     "copy-on-write of partial last blocks on the first step), 256 decode "
                     "steps, one launch over the 1536 items numbered layer-major; inputs "
                     "drawn on the device; no L2 flush")}


def bench_e2e(args, eng, dec, w, n, steps, q, k, v, dq, dk, dv, o_buf, ml_buf, flush, world,
              dist):
    """Same metric through host buffers: Q/K/V of the request and every decode
    step's q/k/v copied in from pinned memory, the kept indices and every
    decode output copied back, all inside the timed events."""
    import torch
    # each decode step's q, k_new, v_new packed in one buffer (host and
    # device), so that a step's inputs arrive with one copy
    def packed(dev_tensors):
        flat = torch.cat([x.reshape(steps, -1).view(torch.uint8) for x in dev_tensors], dim=1)
        views, off = [], 0
        for x in dev_tensors:
            nb = x[0].numel() * 2
            views.append(flat[:, off:off + nb].view(torch.bfloat16).view(x.shape))
            off += nb
        return flat, views
    dqkv_d, (pq, pk, pv) = packed((dq, dk, dv))
    host = {"q": q.cpu().pin_memory(), "k": k.cpu().pin_memory(), "v": v.cpu().pin_memory(),
            "dqkv": dqkv_d.cpu().pin_memory(), "dqkv_d": dqkv_d,
            # one copy stream: host-to-device copies on this machine top out
            # near 211 GB/s whether one or several streams (or a kernel
            # reading pinned memory) move them, and concurrent copies only
            # delay the first layers
            "streams": [torch.cuda.Stream()],
            "out": torch.empty((steps, w.n_layers, w.h_q, w.d), dtype=torch.bfloat16).pin_memory(),
            "kept": torch.empty(n * w.n_layers * w.h_kv, dtype=torch.int32).pin_memory()}
    # untimed warm-up through the host buffers.  Copies out of (and into)
    # pinned memory run at a fraction of the link's rate until the device's
    # translations of its pages are warm: measured on this machine, 17 GB/s on
    # the first pass over a buffer, 34 on the second, 205 from the third on.
    # Freeing large host allocations (a garbage collection after the passes
    # before this one) makes the next pass slow again, so the collection runs
    # first and the collector stays off until the timed requests are done;
    # then three plain copy passes over every host buffer and the warm-up
    # requests.
    gc.collect()
    gc.disable()
    out_d = torch.empty(host["out"].shape, dtype=host["out"].dtype, device=q.device)
    for _ in range(3):
        for hbuf, dbuf in ((host["q"], q), (host["k"], k), (host["v"], v),
                           (host["dqkv"], dqkv_d)):
            dbuf.copy_(hbuf, non_blocking=True)
        host["out"].copy_(out_d, non_blocking=True)
    torch.cuda.synchronize()
    del out_d
    for _ in range(max(1, min(args.warmup, 2))):
        flush()
        run_request(eng, dec, w, n, steps, q, k, v, pq, pk, pv, o_buf, ml_buf, flush,
                    {"prefill": [], "decode": [], "k1": None}, host=host)
    torch.cuda.synchronize()
    rec = {"prefill": [], "decode": [], "k1": None}
    # ten requests, the median of each phase (one request's copies can still
    # meet cold page translations; the per-request prefill times are reported)
    reps = 10
    for _ in range(reps):
        flush()
        run_request(eng, dec, w, n, steps, q, k, v, pq, pk, pv, o_buf, ml_buf, flush, rec,
                    host=host)
    torch.cuda.synchronize()
    gc.enable()
    pre_ms = [a.elapsed_time(b) for a, b in rec["prefill"]]
    dec_ms = [sum(a.elapsed_time(b) for a, b in rec["decode"][i * steps:(i + 1) * steps])
              for i in range(reps)]
    t_pre = float(np.median(pre_ms))
    t_dec = float(np.median(dec_ms))
    t_pre, t_dec = max_over_ranks([t_pre, t_dec], world, dist, q.device)
    kept_bytes = sum(w.k_eff(l, n) for l in range(w.n_layers)) * w.h_kv * 4
    h2d = (q.numel() + k.numel() + v.numel()) * 2 + (dq.numel() + dk.numel() + dv.numel()) * 2
    d2h = kept_bytes + steps * w.n_layers * w.h_q * w.d * 2
    pre_rate, dec_rate = job_rates(t_pre, t_dec, world, n, steps)
    return {"value": round(pre_rate, 1), "unit": "tok/s",
            "decode_tok_s": round(dec_rate, 1),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": reps, "statistic": "median over the requests",
            "prefill_ms_per_request": [round(x, 2) for x in pre_ms],
            "value_mean": round(job_rates(float(np.mean(pre_ms)), float(np.mean(dec_ms)), world,
                                          n, steps)[0], 1)}


# ---------------------------------------------------------------------------
# the CPU oracle, timed on a bounded sample of the same workload
# ---------------------------------------------------------------------------
def cpu_baseline(args):
    """The oracle (fp64 numpy, one thread) on the host cores: prefill rows,
    window scores, selection and compaction of one budgeted layer (all 4000
    rows), and the decode of one step over all 32 layers; scaled to the
    request (x32 layers for prefill+sparsify, per token for decode)."""
    import oracle
    from oracle import flow
    from synth import decode_qkv, llama3_8b, prefill_qkv
    w = llama3_8b()
    n, L = w.prompt_lens[0], w.n_layers
    layer = 3
    rows = np.arange(0, n, max(1, n // args.cpu_rows)) if args.cpu_rows < n else None
    qb, kb, vb = prefill_qkv(w, 0, layer, n)
    t0 = time.perf_counter()
    rec = flow.sparsify_layer(w, layer, qb, kb, vb, rows=rows if rows is not None else np.arange(n))
    pool = oracle.BlockPool(4096)
    pk = np.zeros((4096, w.h_kv, 16, w.d), np.uint16)
    pv = np.zeros_like(pk)
    flow.place_layer(rec, pool, kb, vb, pk, pv)
    t_layer = time.perf_counter() - t0
    frac_rows = (len(rows) if rows is not None else n) / n
    # prefill cost scales with the rows evaluated; the rest is per layer
    t_req_prefill = t_layer / frac_rows * L
    # decode: one step, all layers (caches gathered from the pool)
    recs = []
    for l in range(L):
        k_eff = w.k_eff(l, n)
        r2 = flow.LayerRecord(budgeted=False, k_eff=k_eff,
                              idx=np.tile(np.arange(n - k_eff, n), (w.h_kv, 1)))
        flow.place_layer(r2, pool, kb, vb, pk, pv)
        recs.append(r2)
    st = flow.new_stream(recs)
    dq = [decode_qkv(w, 0, l, 1) for l in range(L)]
    t0 = time.perf_counter()
    for l in range(L):
        flow.prepare_append(pool, st, l, pk, pv)
        flow.append_and_attend(w, st, l, dq[l][0][0], dq[l][1][0], dq[l][2][0], pk, pv)
    t_dec = time.perf_counter() - t0
    return {"value": round(n / t_req_prefill, 3), "unit": "tok/s",
            "decode_tok_s": round(1.0 / t_dec, 3), "cores": 1, "kind": "oracle",
            "sample": (f"layer {layer} of {L}: prefill rows "
                       f"{len(rows) if rows is not None else n}/{n} + scores + selection + "
                       f"compaction, scaled to all rows and 32 layers; decode: one step over "
                       f"32 layers"),
            "host_cores_available": len(os.sched_getaffinity(0))}


def _cpu_unit_worker(layer, dec_layers, rows, start, results):
    """One host core's share of the parallel oracle figure: the prefill +
    sparsify sample of one budgeted layer, then one decode step over its share
    of the 32 layers.  Inputs are drawn before the barrier, so only the
    oracle's work is timed."""
    import oracle
    from oracle import flow
    from synth import decode_qkv, llama3_8b, prefill_qkv
    w = llama3_8b()
    n = w.prompt_lens[0]
    qb, kb, vb = prefill_qkv(w, 0, layer, n)
    dq = [decode_qkv(w, 0, l, 1) for l in dec_layers]
    n_blocks = sum(oracle.blocks_for(w.k_eff(l, n) + 1) for l in dec_layers) + 16
    n_blocks = max(n_blocks, oracle.blocks_for(w.k_eff(layer, n)) + 16)
    start.wait()
    t0 = time.perf_counter()
    rec = flow.sparsify_layer(w, layer, qb, kb, vb, rows=rows)
    pool = oracle.BlockPool(n_blocks)
    pk = np.zeros((n_blocks, w.h_kv, 16, w.d), np.uint16)
    pv = np.zeros_like(pk)
    flow.place_layer(rec, pool, kb, vb, pk, pv)
    t_pre = time.perf_counter() - t0
    # decode caches of this share's layers (set-up, untimed), then one step
    pool = oracle.BlockPool(n_blocks)
    recs = []
    for l in dec_layers:
        k_eff = w.k_eff(l, n)
        r2 = flow.LayerRecord(budgeted=False, k_eff=k_eff,
                              idx=np.tile(np.arange(n - k_eff, n), (w.h_kv, 1)))
        flow.place_layer(r2, pool, kb, vb, pk, pv)
        recs.append(r2)
    st = flow.new_stream(recs)
    start.wait()
    t0 = time.perf_counter()
    for i in range(len(dec_layers)):
        flow.prepare_append(pool, st, i, pk, pv)
        flow.append_and_attend(w, st, i, dq[i][0][0], dq[i][1][0], dq[i][2][0], pk, pv)
    results.put((t_pre, time.perf_counter() - t0))


def cpu_baseline_parallel(args):
    """The same oracle, one process per host core over independent units:
    each process runs one budgeted layer's prefill + sparsify sample (the
    single-core figure's rows), and the 32 layers of one decode step are split
    across the processes.  Processes are spawned (this runs after CUDA work)
    and start together from a barrier; a phase's time is the slowest
    process's.  Prefill+sparsify is scaled as in the single-core figure: the
    P layers done in parallel stand for P of the 32."""
    import multiprocessing as mp
    from synth import llama3_8b
    w = llama3_8b()
    n, L = w.prompt_lens[0], w.n_layers
    P = max(1, min(len(os.sched_getaffinity(0)), L - 3))
    rows = np.arange(0, n, max(1, n // args.cpu_rows)) if args.cpu_rows < n else np.arange(n)
    ctx = mp.get_context("spawn")
    start = ctx.Barrier(P)
    results = ctx.Queue()
    shares = [list(range(i, L, P)) for i in range(P)]
    procs = [ctx.Process(target=_cpu_unit_worker, args=(3 + i, shares[i], rows, start, results))
             for i in range(P)]
    for pr in procs:
        pr.start()
    got = [results.get(timeout=600) for _ in range(P)]
    for pr in procs:
        pr.join(timeout=60)
    t_pre = max(g[0] for g in got)
    t_dec = max(g[1] for g in got)
    t_req_prefill = t_pre / (len(rows) / n) * L / P
    return {"value": round(n / t_req_prefill, 3), "unit": "tok/s",
            "decode_tok_s": round(1.0 / t_dec, 3), "cores": P, "kind": "oracle",
            "sample": (f"{P} processes: layers 3-{2 + P}, each prefill rows {len(rows)}/{n} + "
                       f"scores + selection + compaction, scaled to all rows and 32 layers; "
                       f"decode: one step over 32 layers split across the processes")}


def bench_reference(args):
    """--impl reference: the CPU oracle as the reference arm, on rank 0."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    t0 = time.perf_counter()
    # the oracle on the host's cores (one process per core over independent
    # layers), with the single-core figure beside it
    cb = cpu_baseline_parallel(args)
    one = cpu_baseline(args)
    wall = time.perf_counter() - t0
    out = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "tok/s",
           "decode": {"value": cb["decode_tok_s"], "unit": "tok/s"},
           "n_gpus": 1, "steps": 1, "warmup": 0, "higher_is_better": True,
           "config": {"workload": WORKLOAD}, "dtype": "f64", "data": "synthetic",
           "cpu_baseline": {"value": cb["value"], "unit": "tok/s", "cores": cb["cores"],
                            "kind": "oracle", "sample": cb["sample"],
                            "single_core": {"value": one["value"],
                                            "decode_tok_s": one["decode_tok_s"],
                                            "cores": 1, "sample": one["sample"]}},
           "e2e": {"value": cb["value"], "unit": "tok/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "wall_s": round(wall, 2)}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kvs", choices=["kvs", "reference"])
    ap.add_argument("--decode-steps", type=int, default=500)
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-decode-wall", dest="decode_wall", action="store_false",
                    help="skip the back-to-back decode pass timed by the host clock")
    ap.add_argument("--no-decode-evicting", dest="decode_evicting", action="store_false",
                    help="skip the decode pass with decode-time replacement")
    ap.add_argument("--no-decode-fp8", dest="decode_fp8", action="store_false",
                    help="skip the decode pass over FP8 pools")
    ap.add_argument("--no-decode-per-layer", dest="decode_per_layer", action="store_false",
                    help="skip the model-order decode pass (one launch per layer)")
    ap.add_argument("--no-prefill-per-layer", dest="prefill_per_layer", action="store_false",
                    help="skip the prefill pass with one attention launch per layer")
    ap.add_argument("--no-c2", dest="c2", action="store_false",
                    help="skip the continuous-batching serving pass")
    ap.add_argument("--no-c3", dest="c3", action="store_false",
                    help="skip the long-context pass")
    ap.add_argument("--no-c4", dest="c4", action="store_false",
                    help="skip the shared-prefix pass")
    ap.add_argument("--cpu-rows", type=int, default=400,
                    help="prefill rows the CPU oracle evaluates (sample size)")
    args = ap.parse_args()
    if args.impl == "reference":
        bench_reference(args)
        return
    bench_gpu(args)


if __name__ == "__main__":
    main()
