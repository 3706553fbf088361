"""The algorithmic counts behind the bench's rooflines, at the 4000-token
Llama-3-8B workload, against the sizes the workload's definition gives by
hand: causal prefill flops and exponentials, the kept token-layers after the
per-layer budgets, and the decode bytes per step."""
import bench
from synth import llama3_8b


def test_prefill_counts():
    w, n = llama3_8b(), 4000
    # 2 (QK^T and PV) x 2 flop x d per (head, query, visible key), n(n+1)/2 visible pairs
    per_layer = 2 * 2 * w.d * w.h_q * n * (n + 1) / 2
    assert bench.prefill_flops(w, n) == per_layer
    assert abs(per_layer * w.n_layers - 4.195e12) < 0.001e12
    assert bench.prefill_exps(w, n) == w.h_q * n * (n + 1) / 2


def test_kept_tokens_and_decode_bytes():
    w, n, steps = llama3_8b(), 4000, 500
    keff = [w.k_eff(l, n) for l in range(w.n_layers)]
    # layers 0-2 keep 4000; layer l >= 3 keeps 2048 - 64 (l - 3)
    assert keff[:3] == [4000] * 3 and keff[3] == 2048 and keff[31] == 256
    assert sum(keff) == 45408
    row = w.h_kv * w.d * 2 * 2                       # K and V, bf16, per token and layer
    assert row == 4096
    # one decode launch at the mean length over the request: every cached row
    # (the new one included) read once, plus q, out and the new rows
    lens = [k + steps // 2 for k in keff]
    kv = sum((L + 1) * row for L in lens)
    extra = w.n_layers * (w.h_q * w.d * 2 * 2 + w.h_kv * w.d * 2 * 2)
    assert bench.decode_bytes(w, lens) == kv + extra == 219545600


def test_parallel_oracle_figure_runs_one_process_per_core():
    """The per-core oracle figure spawns one process per host core (at most
    the 29 budgeted layers), each on its own layer, and reports positive
    rates; a small row sample keeps it to a few seconds."""
    import argparse
    import os
    out = bench.cpu_baseline_parallel(argparse.Namespace(cpu_rows=40))
    assert out["cores"] == max(1, min(len(os.sched_getaffinity(0)), 29))
    assert out["kind"] == "oracle" and out["value"] > 0 and out["decode_tok_s"] > 0
