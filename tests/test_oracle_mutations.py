"""Plant plausible mistakes in the oracle (CPU only) and check a pin catches each.

A pin suite that passes on a wrong oracle proves nothing; here each mutant
replaces one oracle step with a subtly wrong version (dropped term, wrong
index, wrong divisor, wrong tie rule ...) and the listed pin tests must fail.
"""

import math

import numpy as np
import pytest

import oracle
from oracle import specprefill_oracle as so
from tests import test_oracle_pins as pins


def _rows_unnormalised(q_bits, k_bits, start, n, layer, kv_head, group, scale=None):
    d = q_bits.shape[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    keys = so.decode_bf16(k_bits[layer, start:start + n, kv_head, :])
    queries = so.decode_bf16(q_bits[layer, :, kv_head * group:(kv_head + 1) * group, :])
    s = np.einsum("lgd,td->lgt", queries, keys) * scale
    return np.exp(s - s.max(axis=-1, keepdims=True))  # mistake: no division by the sum


def _rows_wrong_kv_map(q_bits, k_bits, start, n, layer, kv_head, group, scale=None):
    # mistake: query head h reads KV head h % Hk instead of h // G
    d = q_bits.shape[-1]
    hk = k_bits.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    rows = []
    for j in range(group):
        h = kv_head * group + j
        keys = so.decode_bf16(k_bits[layer, start:start + n, h % hk, :])
        qs = so.decode_bf16(q_bits[layer, :, h, :])
        s = qs @ keys.T * scale
        e = np.exp(s - s.max(axis=-1, keepdims=True))
        rows.append(e / e.sum(axis=-1, keepdims=True))
    return np.stack(rows, axis=1)


def _importance_max_over_steps(step_max):
    return step_max.max(axis=0)  # mistake: max instead of mean over steps


def _pool_fixed_divisor(imp, width):
    half = width // 2
    padded = np.concatenate([np.zeros(half), imp, np.zeros(half)])
    return np.lib.stride_tricks.sliding_window_view(padded, width).sum(axis=1) / width


def _boost_off_by_one(x, first_mult, first_n, last_mult, last_n):
    y = x.copy()
    t = np.arange(y.shape[0])
    y[t <= first_n] *= so.as_f32(first_mult)  # mistake: <= instead of <
    y[t >= y.shape[0] - last_n] *= so.as_f32(last_mult)
    return y


def _rank_ties_descending(cs):
    idx = np.arange(cs.shape[0])
    return np.lexsort((-idx, -cs))  # mistake: ties by descending index


def _mass_without_crossing(cs, mass):
    nc = cs.shape[0]
    sel = np.zeros(nc, dtype=bool)
    total = float(np.sum(cs))
    if not total > 0.0:
        sel[:] = True
        return sel
    theta = so.as_f32(mass) * total
    cum = 0.0
    for c in so.rank_order(cs):
        if cum + cs[c] >= theta:
            break  # mistake: the crossing chunk is dropped
        sel[c] = True
        cum += float(cs[c])
    return sel


def _chunk_means_full_divisor(x, chunk):
    n = x.shape[0]
    nc = (n + chunk - 1) // chunk
    return np.array([x[c * chunk:(c + 1) * chunk].sum() / chunk for c in range(nc)])


def _normalize_no_shift(x):
    lo, hi = x.min(), x.max()
    if hi == lo:
        return np.ones_like(x)
    return x / (hi - lo)  # mistake: the minimum is not subtracted


def _keep_count_float64(nc, keep_p):
    return max(1, int(math.ceil(nc * so.as_f32(keep_p))))  # mistake: float64 product


def _forced_without_tail(n):
    return [t for t in (0, 1, 2, 3) if t < n]  # mistake: n-2 and n-1 dropped


def _eff_min_wrong_divisor(n, min_tok):
    return min(int(min_tok), max(4, n // 100))  # mistake: n / 100


def _cap_without_last(kept, max_keep):
    kept = list(kept)
    if max_keep <= 0 or len(kept) <= max_keep:
        return kept
    step = len(kept) // max_keep
    return kept[::step][:max_keep]  # mistake: the last token is not put back


def _plan_without_break(n, window, stride):
    plan, pos = [], 0
    while pos < n:  # mistake: the loop runs on after the window that reaches the end
        end = min(pos + window, n)
        last = end >= n
        plan.append((pos, end, (end - pos) if last else stride))
        pos += stride
    return plan


def _auto_window_clamp_order(spec_ctx, window=0):
    max_safe = (500 * 1024 * 1024) // (spec_ctx * 32)
    if window <= 0:
        window = min(spec_ctx - 512, max_safe)
    window = min(window, spec_ctx - 128)
    window = max(window, 512)  # mistake: the lower bound applied last
    return window, window // 2


def _pool_rows_fixed_divisor(p, width):
    half = width // 2
    n = p.shape[-1]
    padded = np.concatenate([np.zeros(p.shape[:-1] + (half,)), p, np.zeros(p.shape[:-1] + (half,))], axis=-1)
    return sum(padded[..., o:o + n] for o in range(width)) / width  # mistake: zero padding counted


_STEP_IMPORTANCE = so.step_importance  # the unmutated step, for the mutant that wraps it


def _step_importance_pool_after_max(q_bits, k_bits, start, n, n_kv_heads, scale=None, head_pool_w=1):
    a = _STEP_IMPORTANCE(q_bits, k_bits, start, n, n_kv_heads, scale, 1)
    return so.pool_rows(a, head_pool_w) if head_pool_w > 1 else a  # mistake: pooled after the max


def _run_pins(names):
    failures = 0
    for name in names:
        fn = getattr(pins, name)
        try:
            if name in ("test_oracle_matches_bruteforce", "test_head_pooling_matches_bruteforce"):
                for i in range(len(pins.TINY_CASES)):
                    fn(i)
            elif name == "test_selection_matches_subset_enumeration":
                for seed in range(12):
                    fn(seed)
            else:
                fn()
        except AssertionError:
            failures += 1
    return failures


MUTANTS = [
    ("attention_rows", _rows_unnormalised, ["test_oracle_matches_bruteforce",
                                            "test_softmax_rows_sum_to_one_and_importance_bounds"]),
    ("attention_rows", _rows_wrong_kv_map, ["test_oracle_matches_bruteforce"]),
    ("token_importance", _importance_max_over_steps, ["test_oracle_matches_bruteforce"]),
    ("avg_pool", _pool_fixed_divisor, ["test_pool_properties", "test_oracle_matches_bruteforce"]),
    ("structural_boost", _boost_off_by_one, ["test_boost_positions", "test_oracle_matches_bruteforce"]),
    ("rank_order", _rank_ties_descending, ["test_uniform_attention_gives_equal_chunks",
                                          "test_selection_matches_subset_enumeration"]),
    ("select_mass", _mass_without_crossing, ["test_mass_extremes",
                                            "test_selection_matches_subset_enumeration"]),
    ("chunk_means", _chunk_means_full_divisor, ["test_oracle_matches_bruteforce"]),
    ("min_max_normalize", _normalize_no_shift, ["test_normalize_closed_form",
                                               "test_oracle_matches_bruteforce"]),
    ("listing_keep_count", _keep_count_float64, ["test_listing_keep_count_rounds_the_product_in_float32"]),
    ("listing_forced_tokens", _forced_without_tail, ["test_listing_forced_tokens_and_eff_min",
                                                     "test_listing_ties_keep_every_chunk_at_the_threshold"]),
    ("listing_eff_min", _eff_min_wrong_divisor, ["test_listing_forced_tokens_and_eff_min",
                                                 "test_listing_fill_up_to_eff_min"]),
    ("listing_cap", _cap_without_last, ["test_listing_cap_hand_worked",
                                        "test_listing_keep_all_cases_and_cap"]),
    ("window_plan", _plan_without_break, ["test_window_plan_matches_the_guides_examples",
                                          "test_window_plan_covers_every_token_once"]),
    ("auto_window", _auto_window_clamp_order, ["test_auto_window_closed_forms"]),
    ("pool_rows", _pool_rows_fixed_divisor, ["test_head_pooling_matches_bruteforce",
                                             "test_pool_rows_against_convolution"]),
    ("step_importance", _step_importance_pool_after_max, ["test_head_pooling_matches_bruteforce"]),
]


@pytest.mark.parametrize("target,mutant,pin_names", MUTANTS,
                         ids=[f"{t}:{m.__name__}" for t, m, _ in MUTANTS])
def test_pins_catch_mutant(monkeypatch, target, mutant, pin_names):
    monkeypatch.setattr(so, target, mutant)
    if hasattr(oracle, target):
        monkeypatch.setattr(oracle, target, mutant)
    assert _run_pins(pin_names) >= 1, f"no pin caught the mutant {mutant.__name__}"
