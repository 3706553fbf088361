"""The pins catch plausible mistakes: each test here plants one mistake in the
oracle (a mutated copy of one function, patched in on the CPU for the length
of the test) and checks that the pin meant to catch it then fails.  Nothing
here touches a GPU or the CUDA library."""
import os

import numpy as np
import pytest

import oracle
from oracle import eviction, flow
import test_oracle_pins as pins

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _fails(fn, *args):
    with pytest.raises(AssertionError):
        fn(*args)


# --------------------------------------------------------------------------- selection
def _select_ties_high(scores, n, k, recent):
    if k is None or k >= n:
        return np.arange(n, dtype=np.int64)
    cand = np.arange(0, n - recent)
    order = cand[np.lexsort((-cand, -np.asarray(scores)[cand].astype(np.float64)))]
    return np.sort(np.concatenate([order[: k - recent], np.arange(n - recent, n)]))


def _select_one_too_many(scores, n, k, recent):
    if k is None or k >= n:
        return np.arange(n, dtype=np.int64)
    cand = np.arange(0, n - recent)
    order = cand[np.lexsort((cand, -np.asarray(scores)[cand].astype(np.float64)))]
    return np.sort(np.concatenate([order[: k - recent + 1], np.arange(n - recent, n)]))


def _select_recent_short(scores, n, k, recent):
    if k is None or k >= n:
        return np.arange(n, dtype=np.int64)
    r = max(recent - 1, 0)
    cand = np.arange(0, n - r)
    order = cand[np.lexsort((cand, -np.asarray(scores)[cand].astype(np.float64)))]
    return np.sort(np.concatenate([order[: k - r], np.arange(n - r, n)]))


@pytest.mark.parametrize("mutant", [_select_ties_high, _select_one_too_many, _select_recent_short])
def test_selection_mutants_fail_the_pins(monkeypatch, mutant):
    monkeypatch.setattr(oracle, "select_kept", mutant)
    with pytest.raises(AssertionError):
        pins.test_selection_all_equal_keeps_lowest_positions_and_recent()
        for trial in range(12):
            pins.test_selection_brute_force(trial)


# --------------------------------------------------------------------------- prefill
def _prefill_gqa_modulo(q, k, v, scale, rows=None, heads=None):
    n, h_q, d = q.shape
    h_kv = k.shape[1]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    out = np.zeros((rows.size, h_q, d))
    visible = np.arange(n)[None, :] <= rows[:, None]
    m_out, l_out = np.zeros((h_q, rows.size)), np.zeros((h_q, rows.size))
    for g in range(h_q):
        h = g % h_kv                                    # the mistake: interleaved groups
        s = np.where(visible, (q[rows, g] @ k[:, h].T) * scale, -np.inf)
        m = s.max(axis=1)
        e = np.exp(s - m[:, None])
        out[:, g] = (e / e.sum(axis=1)[:, None]) @ v[:, h]
        m_out[g], l_out[g] = m, e.sum(axis=1)
    return out, m_out, l_out


def _prefill_strict_causal(q, k, v, scale, rows=None, heads=None):
    n, h_q, d = q.shape
    group = h_q // k.shape[1]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    out = np.zeros((rows.size, h_q, d))
    visible = np.arange(n)[None, :] < rows[:, None]      # the mistake: < for <=
    m_out, l_out = np.zeros((h_q, rows.size)), np.zeros((h_q, rows.size))
    with np.errstate(invalid="ignore", divide="ignore"):
        for g in range(h_q):
            h = g // group
            s = np.where(visible, (q[rows, g] @ k[:, h].T) * scale, -np.inf)
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            out[:, g] = (e / e.sum(axis=1)[:, None]) @ v[:, h]
            m_out[g], l_out[g] = m, e.sum(axis=1)
    return out, m_out, l_out


@pytest.mark.parametrize("mutant", [_prefill_gqa_modulo, _prefill_strict_causal])
def test_prefill_mutants_fail_the_pins(monkeypatch, mutant):
    monkeypatch.setattr(oracle, "prefill_rows", mutant)
    _fails(pins.test_prefill_O_equals_sdpa, 67, 4, 2, 16)


# --------------------------------------------------------------------------- window scores
def _scores_window_shifted(q, k, m, l, alpha, scale):
    n, h_q, _ = q.shape
    h_kv = k.shape[1]
    group = h_q // h_kv
    win = np.arange(n - alpha - 1, n - 1)               # the mistake: one row early
    visible = np.arange(n)[None, :] <= win[:, None]
    S = np.zeros((h_kv, n))
    for g in range(h_q):
        s = (q[win, g] @ k[:, g // group].T) * scale
        S[g // group] += (np.exp(np.where(visible, s, -np.inf) - m[g][:, None]) /
                          l[g][:, None]).sum(axis=0)
    return S


def _scores_no_group_sum(q, k, m, l, alpha, scale):
    n, h_q, _ = q.shape
    h_kv = k.shape[1]
    group = h_q // h_kv
    win = np.arange(n - alpha, n)
    visible = np.arange(n)[None, :] <= win[:, None]
    S = np.zeros((h_kv, n))
    for h in range(h_kv):
        g = h * group                                   # the mistake: one query head per group
        s = (q[win, g] @ k[:, h].T) * scale
        S[h] += (np.exp(np.where(visible, s, -np.inf) - m[g][:, None]) /
                 l[g][:, None]).sum(axis=0)
    return S


@pytest.mark.parametrize("mutant", [_scores_window_shifted, _scores_no_group_sum])
def test_window_score_mutants_fail_the_pins(monkeypatch, mutant):
    monkeypatch.setattr(oracle, "window_scores", mutant)
    _fails(pins.test_window_scores_equal_sdpa_probability_column_sums)


# --------------------------------------------------------------------------- paging
class _LifoPool(oracle.BlockPool):
    def alloc(self):
        if not self.free:
            raise oracle.OutOfBlocks()
        b = self.free.pop()                             # the mistake: pop the tail
        self.ref[b] = 1
        return b


def test_lifo_pool_fails_the_worked_example(monkeypatch):
    monkeypatch.setattr(oracle, "BlockPool", _LifoPool)
    _fails(pins.test_paging_worked_example, GOLDEN)


def _compact_ignores_idx(k, v, idx, table, pool_k, pool_v, block=16):
    h_kv, k_eff = idx.shape
    for h in range(h_kv):
        for j in range(k_eff):
            b = table[j // block]
            pool_k[b, h, j % block] = k[j, h]              # the mistake: slot j <- row j
            pool_v[b, h, j % block] = v[j, h]


def _compact_head0_idx(k, v, idx, table, pool_k, pool_v, block=16):
    h_kv, k_eff = idx.shape
    for h in range(h_kv):
        for j in range(k_eff):
            b = table[j // block]
            pool_k[b, h, j % block] = k[idx[0, j], h]      # the mistake: head 0's index
            pool_v[b, h, j % block] = v[idx[0, j], h]


def _compact_sorted_idx(k, v, idx, table, pool_k, pool_v, block=16):
    h_kv, k_eff = idx.shape
    for h in range(h_kv):
        order = np.sort(idx[h])                            # the mistake: index order dropped
        for j in range(k_eff):
            b = table[j // block]
            pool_k[b, h, j % block] = k[order[j], h]
            pool_v[b, h, j % block] = v[order[j], h]


@pytest.mark.parametrize("mutant", [_compact_ignores_idx, _compact_head0_idx, _compact_sorted_idx])
def test_compaction_mutants_fail_the_selected_set_pin(monkeypatch, mutant):
    monkeypatch.setattr(oracle, "compact", mutant)
    _fails(pins.test_compaction_of_a_selected_set_follows_the_index_per_head)


class _PrefixNoParent(oracle.BlockPool):
    def prefix_block(self, layer, parent, tokens):
        return super().prefix_block(layer, -1, tokens)   # the mistake: the prefix is ignored


class _PrefixNoLayer(oracle.BlockPool):
    def prefix_block(self, layer, parent, tokens):
        return super().prefix_block(0, parent, tokens)   # the mistake: layers share keys


class _PrefixNeverForgets(oracle.BlockPool):
    def decref(self, b):
        if self.ref[b] <= 0:
            raise ValueError("decref of a free block")
        self.ref[b] -= 1
        if self.ref[b] == 0:                             # the mistake: the key stays
            self.free.append(b)


@pytest.mark.parametrize("mutant", [_PrefixNoParent, _PrefixNoLayer, _PrefixNeverForgets])
def test_prefix_block_mutants_fail_the_pins(monkeypatch, mutant):
    monkeypatch.setattr(oracle, "BlockPool", mutant)
    with pytest.raises(AssertionError):
        pins.test_prefix_blocks_forgotten_when_free_and_separate_per_layer()
        for seed in range(6):
            pins.test_prefix_blocks_shared_iff_prefixes_equal_brute_force(seed)


# --------------------------------------------------------------------------- decode
def _decode_values_reversed(q, k_cache, v_cache, scale):
    return oracle.attention.decode_attention(q, k_cache, v_cache[:, ::-1], scale)


def test_decode_mutant_fails_the_dense_pin(monkeypatch):
    monkeypatch.setattr(flow, "decode_attention", _decode_values_reversed)
    _fails(pins.test_decode_full_cache_equals_dense_attention)


# --------------------------------------------------------------------------- eviction
def _replace_highest(score, pos, new_pos, recent):
    best = None
    for i in range(len(pos)):
        if pos[i] > new_pos - recent:
            continue
        if best is None or (score[i], -pos[i]) > (score[best], -pos[best]):
            best = i
    return best


def _replace_ignores_window(score, pos, new_pos, recent):
    return int(np.lexsort((pos, score))[0])             # the mistake: recent tokens eligible


@pytest.mark.parametrize("mutant", [_replace_highest, _replace_ignores_window])
def test_eviction_mutants_fail_the_pins(monkeypatch, mutant):
    monkeypatch.setattr(eviction, "replace_slot", mutant)
    _fails(pins.test_eviction_replaces_lowest_outside_recent_window_brute_force)


def _step_variant(score_reset=True, group_sum=True, after_placement=True):
    """A decode step with one of three mistakes: the replaced slot keeps its
    old score, the step's probabilities are averaged over the query group
    instead of summed, or the query attends over the cache as it was before
    the new row was placed."""
    def step(heads, q, k_new, v_new, new_pos, recent, scale, slots=None):
        h_q, d = q.shape
        group = h_q // len(heads)
        before = [(hc.k.copy(), hc.v.copy()) for hc in heads]
        used = []
        for h, hc in enumerate(heads):
            s = eviction.replace_slot(hc.score, hc.pos, new_pos, recent) if slots is None \
                else int(slots[h])
            hc.k[s], hc.v[s], hc.pos[s] = k_new[h], v_new[h], new_pos
            if score_reset:
                hc.score[s] = 0.0
            used.append(s)
        out = np.zeros((h_q, d))
        probs = np.zeros((len(heads), heads[0].k.shape[0]))
        for g in range(h_q):
            hc = heads[g // group]
            kc, vc = (hc.k, hc.v) if after_placement else before[g // group]
            lg = (kc @ q[g]) * scale
            e = np.exp(lg - lg.max())
            pr = e / e.sum()
            out[g] = pr @ vc
            probs[g // group] += pr if group_sum else pr / group
        for h, hc in enumerate(heads):
            hc.score += probs[h]
        return out, probs, used
    return step


@pytest.mark.parametrize("mutant,pin", [
    (_step_variant(score_reset=False),
     pins.test_eviction_replaces_lowest_outside_recent_window_brute_force),
    (_step_variant(group_sum=False), pins.test_eviction_step_attention_is_sdpa_over_the_cache),
    (_step_variant(after_placement=False),
     pins.test_eviction_step_attention_is_sdpa_over_the_cache),
])
def test_eviction_step_mutants_fail_the_pins(monkeypatch, mutant, pin):
    monkeypatch.setattr(eviction, "step", mutant)
    _fails(pin)


def test_eviction_step_variant_without_mistakes_passes_the_pins(monkeypatch):
    # the variant itself, with no mistake switched on, is the oracle's step
    monkeypatch.setattr(eviction, "step", _step_variant())
    pins.test_eviction_step_attention_is_sdpa_over_the_cache()
    pins.test_eviction_replaces_lowest_outside_recent_window_brute_force()


# --------------------------------------------------------------------------- FP8
def _encode_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    vals = oracle.fp8.E4M3_TABLE[:0x7F]
    sign = np.where(np.signbit(x), 0x80, 0)
    a = np.minimum(np.abs(x), 448.0)
    lo = np.clip(np.searchsorted(vals, a, side="right") - 1, 0, 126)
    hi = np.minimum(lo + 1, 126)
    pick_lo = (a - vals[lo]) < (vals[hi] - a)           # the mistake: ties go up
    return (sign | np.where(pick_lo, lo, hi)).astype(np.uint8)


def _value_bias_8(code):
    code = int(code) & 0xFF
    if code in (0x7F, 0xFF):
        return float("nan")
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 8)      # the mistake: bias 8


def _quantize_scale_447(x):
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.abs(x32).max())
    scale = np.float32(amax / np.float32(447.0)) if amax > 0 else np.float32(1.0)
    return oracle.fp8.e4m3_encode((x32 / scale).astype(np.float32)), scale


def test_fp8_encode_mutant_fails_the_torch_pin(monkeypatch):
    monkeypatch.setattr(oracle.fp8, "e4m3_encode", _encode_ties_away)
    _fails(pins.test_fp8_encode_matches_torch_round_to_nearest_even)


def test_fp8_decode_mutant_fails_the_torch_pin(monkeypatch):
    monkeypatch.setattr(oracle.fp8, "e4m3_value", _value_bias_8)
    _fails(pins.test_fp8_decode_matches_torch_for_every_code)


def test_fp8_scale_mutant_fails_the_bound_pin(monkeypatch):
    monkeypatch.setattr(oracle.fp8, "quantize_row", _quantize_scale_447)
    _fails(pins.test_fp8_row_quantisation_bounds)
