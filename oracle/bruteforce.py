"""Brute-force twin of the float64 oracle, for tiny inputs only.

TEST INFRASTRUCTURE (same rules as the oracle: tests only). Pure-Python
loops with math.fsum and math.exp, written independently of the vectorised
oracle so that the two can pin each other: every logit is an explicit dot
product, every window sum an explicit loop, and the selection is found by
enumerating all chunk subsets and testing the defining property instead of
walking a sorted order.

Definitions followed (same pages as the oracle):
* importance = mean over lookahead steps of (max over layers and heads of
  the softmax row), "SpecPrefill — Implementation Guide" §How It Works /
  Token Importance;
* W-wide centred average pool, PR "Speculative prefill" §Approach item 3,
  either on the per-token importance or (pool_at = "head") on every softmax
  row before the max over heads and layers;
* min-max normalisation, guide v3.1 §v3.1 Optimizations item 5;
* structural boost, guide v3 §v3 Improvements item 2;
* chunk mean and ranking, guide §Chunk Selection; cumulative mass, guide v3
  §v3 Improvements item 1; BOS and the final chunk always kept, PR §Approach
  item 4.
"""

import itertools
import math
import struct
from typing import Dict, List


def bf16_value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", float(x)))[0]


def _prompt_importance(q, k, start: int, n: int, scale: float, row_pool: int = 1) -> List[float]:
    n_layers, n_steps, n_q_heads, d = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    n_kv_heads = len(k[0][0])
    group = n_q_heads // n_kv_heads
    best = [[-math.inf] * n for _ in range(n_steps)]
    for layer in range(n_layers):
        for h in range(n_q_heads):
            g = h // group
            for s in range(n_steps):
                qv = [bf16_value(v) for v in q[layer][s][h]]
                logits = []
                for t in range(n):
                    kv = [bf16_value(v) for v in k[layer][start + t][g]]
                    logits.append(scale * math.fsum(qv[i] * kv[i] for i in range(d)))
                top = max(logits)
                ex = [math.exp(x - top) for x in logits]
                z = math.fsum(ex)
                row = [ex[t] / z for t in range(n)]
                if row_pool > 1:
                    row = _pool(row, row_pool)
                for t in range(n):
                    if row[t] > best[s][t]:
                        best[s][t] = row[t]
    return [math.fsum(best[s][t] for s in range(n_steps)) / n_steps for t in range(n)]


def _pool(v: List[float], width: int) -> List[float]:
    n, half = len(v), width // 2
    out = []
    for t in range(n):
        window = [v[u] for u in range(t - half, t + half + 1) if 0 <= u < n]
        out.append(math.fsum(window) / len(window))
    return out


def _is_upper_set(subset, cs) -> bool:
    """Every member outranks every non-member (score desc, index asc)."""
    inside = set(subset)
    for i in inside:
        for j in range(len(cs)):
            if j in inside:
                continue
            if not (cs[i] > cs[j] or (cs[i] == cs[j] and i < j)):
                return False
    return True


def _select(cs: List[float], mode: str, keep_p: float, mass: float) -> List[int]:
    nc = len(cs)
    assert nc <= 12, "subset enumeration is for tiny cases only"
    if mode == "fixed":
        k = min(nc, max(1, math.ceil(nc * f32(keep_p))))
        found = [s for s in itertools.combinations(range(nc), k) if _is_upper_set(s, cs)]
        assert len(found) == 1
        return sorted(found[0])
    total = math.fsum(cs)
    if not total > 0:
        return list(range(nc))
    theta = f32(mass) * total
    for size in range(1, nc + 1):
        for s in itertools.combinations(range(nc), size):
            if _is_upper_set(s, cs) and math.fsum(cs[c] for c in s) >= theta:
                return sorted(s)
    return list(range(nc))


def run_bruteforce(q, k, seq_off, *, pool_w=13, chunk=32, mode="fixed", keep_p=0.30,
                   mass=0.85, normalize=True, boost_first_mult=1.5, boost_first_n=64,
                   boost_last_mult=1.3, boost_last_n=128, force_bos=True,
                   force_last_chunk=True, scale=None, select=True,
                   pool_at="token") -> Dict[str, list]:
    """Same outputs as the oracle's ``run`` (lists instead of arrays).

    q: nested [B][Ly][L][Hq][d] bf16 bits; k: nested [Ly][Ntot][Hk][d] bf16 bits.
    """
    q = q.tolist() if hasattr(q, "tolist") else q
    k = k.tolist() if hasattr(k, "tolist") else k
    seq_off = [int(v) for v in seq_off]
    d = len(k[0][0][0])
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = {"imp": [], "tok_score": [], "final_score": [], "chunk_score": [],
           "chunk_keep": [], "kept_idx": [], "kept_pos": [], "kept_off": [0]}
    for b in range(len(seq_off) - 1):
        start, n = seq_off[b], seq_off[b + 1] - seq_off[b]
        imp = _prompt_importance(q[b], k, start, n, scale, pool_w if pool_at == "head" else 1)
        x = _pool(imp, pool_w if pool_at == "token" else 1)
        y = list(x)
        if normalize:
            lo, hi = min(y), max(y)
            y = [1.0] * n if hi == lo else [(v - lo) / (hi - lo) for v in y]
        for t in range(n):
            if t < boost_first_n:
                y[t] = y[t] * f32(boost_first_mult)
            if t >= n - boost_last_n:
                y[t] = y[t] * f32(boost_last_mult)
        nc = -(-n // chunk)
        cs = []
        for c in range(nc):
            members = y[c * chunk:min(n, (c + 1) * chunk)]
            cs.append(math.fsum(members) / len(members))
        out["imp"] += imp
        out["tok_score"] += x
        out["final_score"] += y
        out["chunk_score"] += cs
        if not select:
            continue
        chosen = set(_select(cs, mode, keep_p, mass))
        flags = [(1 if c in chosen else 0) | (2 if (force_last_chunk and c == nc - 1) else 0)
                 for c in range(nc)]
        kept = [t for t in range(n) if flags[t // chunk] or (force_bos and t == 0)]
        out["chunk_keep"] += flags
        out["kept_idx"] += [start + t for t in kept]
        out["kept_pos"] += kept
        out["kept_off"].append(out["kept_off"][-1] + len(kept))
    return out
