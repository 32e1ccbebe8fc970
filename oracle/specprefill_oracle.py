"""Float64 CPU oracle of the SpecPrefill token-importance and chunk-selection path.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg may import this module. The product (the CUDA library and its
binding) never calls it, and it shares no code with that product.

Each function is one step of the method, in the order the pages give it, in
plain numpy float64 (inputs are bf16 bit patterns decoded exactly):

1. logits   s = scale * <q, k>, scale = 1/sqrt(d)            (PR "Speculative
   prefill" §Approach item 2; guide "SpecPrefill — Implementation Guide"
   §Sliding Window / The OOM Problem: the attention matrix is Q @ K^T)
2. softmax  over the prompt's N keys                          (guide §How It
   Works / Attention Capture: post-softmax kq_soft_max rows)
3. max over heads, then max over layers                       (guide §How It
   Works / Token Importance, steps 2-3; listing `compute_imp`)
4. mean over lookahead steps                                  (same section)
5. 1D average pool, W = 13, centred, in-range divisor         (PR §Approach
   item 3)
6. min-max normalisation to [0, 1]                            (guide v3.1,
   §v3.1 Optimizations item 5)
7. structural boost: first 64 tokens x1.5, last 128 x1.3      (guide v3,
   §v3 Improvements item 2)
8. chunk score = mean over a 32-token contiguous chunk        (guide §Chunk
   Selection; listing `select_chunks`)
9-10. rank chunks (score descending, index ascending) and keep either the
   top k = max(1, ceil(nc * p)) or the shortest prefix whose cumulative
   score reaches mass * total                                 (guide v3,
   §v3 Improvements item 1; listing `select_chunks`)
11. force BOS (token 0) and the final chunk                   (PR §Approach
   item 4)
12. kept-token list with original position IDs                (guide §How It
   Works / Sparse Prefill)
13. rows of the kept tokens gathered from a token-major cache
   tensor, in kept-list order, for the target's sparse prefill (same
   section: only the kept tokens are prefilled; listing of the sparse pass
   adds kept[i] with its position to the target batch)

Per-head pooling variant (the PR's other reading of where the smoothing
sits, §Approach item 3: "smoothed ... max-reduced across heads/layers"):
5'. with pool_at = "head", every softmax row p[layer, step, head, :] is
   pooled (the same centred in-range mean, width W) before the max of
   step 3; step 5 is then the identity.

Reference-compatibility variants (the pages' own tool, for A/B comparison):
14. listing selection rule: k = max(1, ceil(nc * p)) with the product in
   float32, every chunk scoring at least the k-th score kept (ties can keep
   more than k), tokens {0, 1, 2, 3, n-2, n-1} forced, a fill up to
   eff_min = min(min_tok, max(4, n // 10)) tokens from the unselected chunks
   in ascending order, everything kept when p >= 1 or n <= eff_min, and a
   strided cap to max_keep tokens that keeps the last one  (guide v2 listing
   `select_chunks` and the cap after it in `main`)
15. sliding-window scoring: windows of `window` tokens every `stride`
   tokens, each contributing its first `stride` scores (the last window all
   of its own), averaged per token; the window size comes from the draft's
   context size                                               (guide v3.1,
   §Sliding Window Loop and §Bug Fixes in v3.1; guide v2 listing `main`,
   window sizing)

In-situ draft caches: a draft engine keeps K per layer in pools of
fixed-size blocks with a per-prompt block table (logical block -> physical
block); kv_from_pages gathers such a cache back into the dense token-major
[Ly, Ntot, Hk, d] layout the steps above read, so the scores of a paged
cache are by definition those of its dense gather.

Readings where the pages are silent (each also listed in the design notes):
softmax over the prompt keys only; kv head = h // G; the pool divides by the
number of in-range tokens and never crosses a prompt boundary; normalisation
of a constant vector gives all ones; boost factors multiply where the two
regions overlap; ties in the ranking break by ascending chunk index and the
fixed mode keeps exactly k chunks; a chunk's mass is its score, the crossing
chunk is kept, forced chunks do not count, and zero total mass keeps all;
forced chunks/tokens are added after the ranking selection; an empty prompt
(zero tokens) has no chunks and keeps nothing.
"""

import math
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence

import numpy as np


# ---------------------------------------------------------------------------
# input decoding


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact float64 values (bf16 is the top half of fp32)."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def as_f32(x: float) -> float:
    """The float64 value of a float32 parameter (p and mass are float32 inputs)."""
    return float(np.float32(x))


# ---------------------------------------------------------------------------
# steps 1-4: attention rows and token importance


def attention_rows(q_bits: np.ndarray, k_bits: np.ndarray, start: int, n: int,
                   layer: int, kv_head: int, group: int,
                   scale: Optional[float] = None) -> np.ndarray:
    """Softmax rows of one (layer, KV head) for one prompt.

    q_bits: [Ly, L, Hq, d] of the prompt; k_bits: [Ly, Ntot, Hk, d].
    Returns p[l, j, t] for lookahead step l, query head h = kv_head*group + j,
    prompt key t in [0, n). Steps 1 and 2.
    """
    d = q_bits.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    keys = decode_bf16(k_bits[layer, start:start + n, kv_head, :])            # [n, d]
    heads = slice(kv_head * group, (kv_head + 1) * group)
    queries = decode_bf16(q_bits[layer, :, heads, :])                           # [L, G, d]
    n_steps = queries.shape[0]
    s = (queries.reshape(-1, d) @ keys.T).reshape(n_steps, group, n) * scale    # step 1
    s_max = s.max(axis=-1, keepdims=True)
    e = np.exp(s - s_max)
    return e / e.sum(axis=-1, keepdims=True)                                     # step 2


def pool_rows(p: np.ndarray, width: int) -> np.ndarray:
    """Centred in-range mean of odd ``width`` along the last axis of every
    row (step 5'): the sum over the window offsets -W/2 .. W/2 of the row
    shifted by that offset (positions outside [0, n) add nothing), divided
    by the number of in-range positions."""
    n = p.shape[-1]
    half = width // 2
    acc = np.zeros_like(p, dtype=np.float64)
    cnt = np.zeros(n, dtype=np.float64)
    for o in range(-half, half + 1):
        lo, hi = max(0, -o), min(n, n - o)     # t with t + o in [0, n)
        if lo >= hi:
            continue
        acc[..., lo:hi] += p[..., lo + o:hi + o]
        cnt[lo:hi] += 1.0
    return acc / cnt


def step_importance(q_bits: np.ndarray, k_bits: np.ndarray, start: int, n: int,
                    n_kv_heads: int, scale: Optional[float] = None,
                    head_pool_w: int = 1) -> np.ndarray:
    """A[l, t] = max over layers and query heads of p (step 3), shape [L, n];
    with head_pool_w > 1 each row is pooled first (step 5')."""
    n_layers, n_steps, n_q_heads, _ = q_bits.shape
    group = n_q_heads // n_kv_heads
    a = np.full((n_steps, n), -np.inf)
    for layer in range(n_layers):
        for g in range(n_kv_heads):
            p = attention_rows(q_bits, k_bits, start, n, layer, g, group, scale)
            if head_pool_w > 1:
                p = pool_rows(p, head_pool_w)
            a = np.maximum(a, p.max(axis=1))
    return a


def token_importance(step_max: np.ndarray) -> np.ndarray:
    """imp[t] = mean over lookahead steps of A[l, t] (step 4)."""
    return step_max.sum(axis=0) / step_max.shape[0]


# ---------------------------------------------------------------------------
# steps 5-8: smoothing, normalisation, boost, chunk scores


def avg_pool(imp: np.ndarray, width: int) -> np.ndarray:
    """Centred moving average of odd ``width``: the mean of the window
    positions inside [0, n) (step 5). Each window sum is exact (math.fsum),
    so windows holding the same tokens give identical means."""
    n = imp.shape[0]
    half = width // 2
    vals = imp.tolist()
    out = np.empty(n)
    for t in range(n):
        lo, hi = max(0, t - half), min(n, t + half + 1)
        out[t] = math.fsum(vals[lo:hi]) / (hi - lo)
    return out


def min_max_normalize(x: np.ndarray) -> np.ndarray:
    """(x - min) / (max - min); a constant vector maps to all ones (step 6)."""
    lo, hi = x.min(), x.max()
    if hi == lo:
        return np.ones_like(x)
    return (x - lo) / (hi - lo)


def structural_boost(x: np.ndarray, first_mult: float, first_n: int,
                     last_mult: float, last_n: int) -> np.ndarray:
    """Multiply positions t < first_n by first_mult, then t >= n - last_n by
    last_mult (step 7). Multipliers are float32 parameters."""
    y = x.copy()
    n = y.shape[0]
    t = np.arange(n)
    y[t < first_n] *= as_f32(first_mult)
    y[t >= n - last_n] *= as_f32(last_mult)
    return y


def chunk_means(x: np.ndarray, chunk: int) -> np.ndarray:
    """Mean score of each contiguous chunk; the last chunk may be partial (step 8)."""
    n = x.shape[0]
    nc = (n + chunk - 1) // chunk
    return np.array([x[c * chunk:min((c + 1) * chunk, n)].mean() for c in range(nc)])


# ---------------------------------------------------------------------------
# steps 9-12: ranking, selection, forcing, kept list


def rank_order(cs: np.ndarray) -> np.ndarray:
    """Chunk indices sorted by score descending, then index ascending (step 9)."""
    idx = np.arange(cs.shape[0])
    return np.lexsort((idx, -cs))


def fixed_count(nc: int, keep_p: float) -> int:
    """k = max(1, ceil(nc * p)), evaluated in float64 on the float32 p."""
    return max(1, int(math.ceil(nc * as_f32(keep_p))))


def select_fixed(cs: np.ndarray, keep_p: float) -> np.ndarray:
    """Boolean mask of the top-k chunks of the ranking (step 10, fixed mode)."""
    order = rank_order(cs)
    k = min(fixed_count(cs.shape[0], keep_p), cs.shape[0])
    sel = np.zeros(cs.shape[0], dtype=bool)
    sel[order[:k]] = True
    return sel


def select_mass(cs: np.ndarray, mass: float) -> np.ndarray:
    """Walk the ranking, keeping chunks until the running sum of their scores
    reaches mass * (sum of all scores); the crossing chunk is kept. Zero total
    mass keeps every chunk (step 10, mass mode)."""
    nc = cs.shape[0]
    sel = np.zeros(nc, dtype=bool)
    total = float(np.sum(cs))
    if not total > 0.0:
        sel[:] = True
        return sel
    theta = as_f32(mass) * total
    cum = 0.0
    for c in rank_order(cs):
        sel[c] = True
        cum += float(cs[c])
        if cum >= theta:
            break
    return sel


@dataclass
class Selection:
    chunk_keep: np.ndarray   # uint8 per chunk: bit0 ranked-selected, bit1 forced final chunk
    kept_tokens: np.ndarray  # int64 sorted token positions within the prompt


def finish_selection(sel: np.ndarray, n: int, chunk: int, force_bos: bool,
                     force_last_chunk: bool) -> Selection:
    """Add the forced final chunk and BOS token, expand chunks to tokens
    (steps 11-12)."""
    nc = sel.shape[0]
    flags = sel.astype(np.uint8)
    if nc == 0:
        return Selection(chunk_keep=flags, kept_tokens=np.zeros(0, dtype=np.int64))
    if force_last_chunk:
        flags[nc - 1] |= 2
    toks: List[int] = []
    for c in range(nc):
        if flags[c]:
            toks.extend(range(c * chunk, min((c + 1) * chunk, n)))
    if force_bos and not flags[0]:
        toks.append(0)
    return Selection(chunk_keep=flags, kept_tokens=np.array(sorted(toks), dtype=np.int64))


# ---------------------------------------------------------------------------
# 14. the listing's selection rule (reference-compatibility mode)


def listing_keep_count(nc: int, keep_p: float) -> int:
    """k = max(1, ceil(nc * p)) where nc * p is an int times a float32, so
    the product is rounded to float32 before the ceiling (5 * 0.4f gives
    2.0, not 2.0000000298)."""
    prod = np.float32(nc) * np.float32(keep_p)
    return max(1, int(math.ceil(float(prod))))


def listing_eff_min(n: int, min_tok: int) -> int:
    """Smallest kept-token count: min(min_tok, max(4, n // 10))."""
    return min(int(min_tok), max(4, n // 10))


def listing_forced_tokens(n: int) -> List[int]:
    """Tokens 0-3 and, when the prompt has more than four, the last two."""
    forced = [t for t in (0, 1, 2, 3) if t < n]
    if n > 4:
        forced += [n - 2, n - 1]
    return sorted(set(forced))


def listing_cap(kept: Sequence[int], max_keep: int) -> List[int]:
    """Keep every step-th entry (step = len // max_keep) up to max_keep
    entries, the last entry replaced by the list's last token; max_keep <= 0
    disables the cap."""
    kept = list(kept)
    if max_keep <= 0 or len(kept) <= max_keep:
        return kept
    step = len(kept) // max_keep
    capped = []
    i = 0
    while i < len(kept) and len(capped) < max_keep:
        capped.append(kept[i])
        i += step
    capped[-1] = kept[-1]
    return capped


def select_listing(cs: np.ndarray, n: int, *, chunk: int, mode: str, keep_p: float,
                   mass: float, min_tok: int, max_keep: int) -> Selection:
    """Steps 9-12 under the listing's rule. Fixed mode keeps every chunk whose
    score is at least the k-th largest; mass mode keeps the ranking prefix of
    step 10. Then the forced tokens, the fill from unselected chunks (chunk
    order, token order) up to eff_min, and the cap. chunk_keep has bit 0 for
    the chunks the ranking (or the keep-everything case) selected."""
    nc = cs.shape[0]
    if n == 0:
        return Selection(chunk_keep=np.zeros(0, dtype=np.uint8), kept_tokens=np.zeros(0, dtype=np.int64))
    eff_min = listing_eff_min(n, min_tok)
    if (mode == "fixed" and as_f32(keep_p) >= 1.0) or n <= eff_min:
        sel = np.ones(nc, dtype=bool)
    elif mode == "fixed":
        kc = listing_keep_count(nc, keep_p)
        ordered = sorted((float(v) for v in cs), reverse=True)
        th = ordered[kc - 1] if kc <= nc else -math.inf
        sel = np.array([float(v) >= th for v in cs], dtype=bool)
    elif mode == "mass":
        sel = select_mass(cs, mass)
    else:
        raise ValueError(mode)
    kept = set()
    for c in range(nc):
        if sel[c]:
            kept.update(range(c * chunk, min((c + 1) * chunk, n)))
    kept.update(listing_forced_tokens(n))
    if len(kept) < eff_min:
        for c in range(nc):
            if len(kept) >= eff_min:
                break
            if sel[c]:
                continue
            for t in range(c * chunk, min((c + 1) * chunk, n)):
                if len(kept) >= eff_min:
                    break
                kept.add(t)
    toks = listing_cap(sorted(kept), max_keep)
    return Selection(chunk_keep=sel.astype(np.uint8), kept_tokens=np.array(toks, dtype=np.int64))


# ---------------------------------------------------------------------------
# 15. sliding-window scoring (reference-compatibility mode)


def auto_window(spec_ctx: int, window: int = 0):
    """(window, stride) for a draft context of spec_ctx tokens: a requested
    window <= 0 becomes min(spec_ctx - 512, 500 MiB / (spec_ctx * 32)); the
    result is clamped to [512, spec_ctx - 128] (upper bound last) and the
    stride is half of it."""
    max_safe = (500 * 1024 * 1024) // (spec_ctx * 32)
    if window <= 0:
        window = min(spec_ctx - 512, max_safe)
    window = max(window, 512)
    window = min(window, spec_ctx - 128)
    return window, window // 2


def window_plan(n: int, window: int, stride: int):
    """Windows of the fixed loop: (start, end, kept) per window, where the
    window scores tokens [start, end) and contributes its first `kept`
    scores; the loop stops after the first window that reaches the end of
    the prompt or whose next start would."""
    if stride < 1 or window < stride:
        raise ValueError("need 1 <= stride <= window")
    plan = []
    pos = 0
    while pos < n:
        end = min(pos + window, n)
        last = end >= n or pos + stride >= n
        plan.append((pos, end, (end - pos) if last else stride))
        if last:
            break
        pos += stride
    return plan


def merge_windows(window_imps: Sequence[np.ndarray], n: int, window: int, stride: int) -> np.ndarray:
    """Per-token average of the window contributions; a token no window
    scored gets 1.0."""
    plan = window_plan(n, window, stride)
    if len(window_imps) != len(plan):
        raise ValueError("one importance vector per window")
    acc = np.zeros(n, dtype=np.float64)
    cnt = np.zeros(n, dtype=np.int64)
    for (start, end, kept), imp in zip(plan, window_imps):
        imp = np.asarray(imp, dtype=np.float64)
        if imp.shape[0] != end - start:
            raise ValueError("window importance has the wrong length")
        for i in range(kept):
            acc[start + i] += imp[i]
            cnt[start + i] += 1
    return np.where(cnt > 0, acc / np.maximum(cnt, 1), 1.0)


# ---------------------------------------------------------------------------
# whole path


def score_prompt(imp: np.ndarray, *, pool_w: int, chunk: int, normalize: bool,
                 boost_first_mult: float, boost_first_n: int,
                 boost_last_mult: float, boost_last_n: int) -> Dict[str, np.ndarray]:
    """Steps 5-8 for one prompt."""
    x = avg_pool(imp, pool_w)
    y = min_max_normalize(x) if normalize else x
    y = structural_boost(y, boost_first_mult, boost_first_n, boost_last_mult, boost_last_n)
    return {"tok_score": x, "final_score": y, "chunk_score": chunk_means(y, chunk)}


def select_prompt(cs: np.ndarray, n: int, *, chunk: int, mode: str, keep_p: float,
                  mass: float, force_bos: bool, force_last_chunk: bool, rule: str = "exact",
                  min_tok: int = 128, max_keep: int = 0) -> Selection:
    """Steps 9-12 for one prompt (rule "listing": step 14 instead)."""
    if rule == "listing":
        return select_listing(cs, n, chunk=chunk, mode=mode, keep_p=keep_p, mass=mass,
                              min_tok=min_tok, max_keep=max_keep)
    if rule != "exact":
        raise ValueError(rule)
    if cs.shape[0] == 0:
        sel = np.zeros(0, dtype=bool)
    elif mode == "fixed":
        sel = select_fixed(cs, keep_p)
    elif mode == "mass":
        sel = select_mass(cs, mass)
    else:
        raise ValueError(mode)
    return finish_selection(sel, n, chunk, force_bos, force_last_chunk)


def chunk_offsets(seq_off: np.ndarray, chunk: int) -> np.ndarray:
    lengths = np.diff(np.asarray(seq_off, dtype=np.int64))
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    out[1:] = np.cumsum((lengths + chunk - 1) // chunk)
    return out


def select_from_chunk_scores(chunk_score: np.ndarray, seq_off: np.ndarray, *, chunk: int,
                             mode: str, keep_p: float, mass: float, force_bos: bool,
                             force_last_chunk: bool, rule: str = "exact", min_tok: int = 128,
                             max_keep: int = 0, **_unused) -> Dict[str, np.ndarray]:
    """Steps 9-12 over a packed batch of given chunk scores."""
    seq_off = np.asarray(seq_off, dtype=np.int64)
    coff = chunk_offsets(seq_off, chunk)
    keep, idx, pos, koff = [], [], [], [0]
    for b in range(len(seq_off) - 1):
        n = int(seq_off[b + 1] - seq_off[b])
        cs = np.asarray(chunk_score[coff[b]:coff[b + 1]], dtype=np.float64)
        s = select_prompt(cs, n, chunk=chunk, mode=mode, keep_p=keep_p, mass=mass,
                          force_bos=force_bos, force_last_chunk=force_last_chunk, rule=rule,
                          min_tok=min_tok, max_keep=max_keep)
        keep.append(s.chunk_keep)
        idx.append(s.kept_tokens + seq_off[b])
        pos.append(s.kept_tokens)
        koff.append(koff[-1] + len(s.kept_tokens))
    return {
        "chunk_off": coff,
        "chunk_keep": np.concatenate(keep),
        "kept_idx": np.concatenate(idx),
        "kept_pos": np.concatenate(pos),
        "kept_off": np.array(koff, dtype=np.int64),
    }


def score_from_importance(imp: np.ndarray, seq_off: Sequence[int], *, pool_w: int = 13,
                          chunk: int = 32, mode: str = "fixed", keep_p: float = 0.30,
                          mass: float = 0.85, normalize: bool = True,
                          boost_first_mult: float = 1.5, boost_first_n: int = 64,
                          boost_last_mult: float = 1.3, boost_last_n: int = 128,
                          force_bos: bool = True, force_last_chunk: bool = True,
                          rule: str = "exact", min_tok: int = 128, max_keep: int = 0,
                          pool_at: str = "token") -> Dict[str, np.ndarray]:
    """Steps 5-12 over a packed batch of per-token importance vectors (with
    pool_at = "head" the importance is already pooled: no step 5)."""
    if pool_at not in ("token", "head"):
        raise ValueError(pool_at)
    if pool_at == "head":
        pool_w = 1
    seq_off = np.asarray(seq_off, dtype=np.int64)
    imp = np.asarray(imp, dtype=np.float64)
    toks, finals, chunks = [], [], []
    for b in range(len(seq_off) - 1):
        start, end = int(seq_off[b]), int(seq_off[b + 1])
        if end == start:
            for lst in (toks, finals, chunks):
                lst.append(np.zeros(0))
            continue
        sc = score_prompt(imp[start:end], pool_w=pool_w, chunk=chunk, normalize=normalize,
                          boost_first_mult=boost_first_mult, boost_first_n=boost_first_n,
                          boost_last_mult=boost_last_mult, boost_last_n=boost_last_n)
        toks.append(sc["tok_score"])
        finals.append(sc["final_score"])
        chunks.append(sc["chunk_score"])
    out = {
        "imp": imp,
        "tok_score": np.concatenate(toks),
        "final_score": np.concatenate(finals),
        "chunk_score": np.concatenate(chunks),
    }
    out.update(select_from_chunk_scores(out["chunk_score"], seq_off, chunk=chunk, mode=mode,
                                        keep_p=keep_p, mass=mass, force_bos=force_bos,
                                        force_last_chunk=force_last_chunk, rule=rule,
                                        min_tok=min_tok, max_keep=max_keep))
    return out


def importance(q_bits: np.ndarray, k_bits: np.ndarray, seq_off: Sequence[int], *,
               scale: Optional[float] = None, keep_step_max: bool = False,
               pool_at: str = "token", pool_w: int = 13):
    """Steps 1-4 over a packed batch: imp per token (and, on request, the
    per-step maxima A[l, t] of each prompt); pool_at = "head" pools every
    softmax row with width pool_w before the max (step 5')."""
    if pool_at not in ("token", "head"):
        raise ValueError(pool_at)
    head_pool_w = pool_w if pool_at == "head" else 1
    seq_off = np.asarray(seq_off, dtype=np.int64)
    n_kv_heads = k_bits.shape[2]
    imps, steps = [], []
    for b in range(len(seq_off) - 1):
        start, n = int(seq_off[b]), int(seq_off[b + 1] - seq_off[b])
        if n == 0:
            imps.append(np.zeros(0))
            steps.append(np.zeros((q_bits.shape[2], 0)))
            continue
        a = step_importance(q_bits[b], k_bits, start, n, n_kv_heads, scale, head_pool_w)
        imps.append(token_importance(a))
        steps.append(a)
    imp = np.concatenate(imps)
    return (imp, steps) if keep_step_max else imp


def run(q_bits: np.ndarray, k_bits: np.ndarray, seq_off: Sequence[int], *,
        scale: Optional[float] = None, keep_step_max: bool = False, **kw) -> Dict[str, np.ndarray]:
    """The whole path over a packed batch.

    q_bits: [B, Ly, L, Hq, d] bf16 bits; k_bits: [Ly, Ntot, Hk, d] bf16 bits;
    seq_off: [B+1] prompt offsets into the token axis of k; the selection
    keywords are those of score_from_importance (defaults: W = 13, C = 32,
    fixed p = 0.30, mass 0.85, normalise, boost 1.5 x 64 / 1.3 x 128, BOS and
    final chunk forced, the exact rule).
    Returns float64 imp / tok_score / final_score (per token), chunk_score and
    chunk_keep (per chunk), and the kept lists (packed index, position,
    per-prompt offsets).
    """
    imp, steps = importance(q_bits, k_bits, seq_off, scale=scale, keep_step_max=True,
                            pool_at=kw.get("pool_at", "token"), pool_w=kw.get("pool_w", 13))
    out = score_from_importance(imp, seq_off, **kw)
    if keep_step_max:
        out["step_max"] = steps
    return out


# ---------------------------------------------------------------------------
# in-situ draft caches


def kv_from_pages(pools: Sequence[np.ndarray], block_table: np.ndarray, seq_off: Sequence[int],
                  block_size: int) -> np.ndarray:
    """Dense token-major keys from per-layer block pools.

    pools: one array per layer, [num_blocks, block_size, Hk, d];
    block_table: [B, max_blocks] physical block of each logical block of
    prompt b; logical token t of prompt b sits in block
    block_table[b, t // block_size] at row t % block_size.
    Returns [Ly, Ntot, Hk, d] with prompt b at tokens seq_off[b] + t.
    """
    seq_off = np.asarray(seq_off, dtype=np.int64)
    ly = len(pools)
    _, bs, hk, d = pools[0].shape
    if bs != block_size:
        raise ValueError("pool block size differs from block_size")
    out = np.zeros((ly, int(seq_off[-1]), hk, d), dtype=pools[0].dtype)
    for layer in range(ly):
        for b in range(len(seq_off) - 1):
            start, n = int(seq_off[b]), int(seq_off[b + 1] - seq_off[b])
            for t in range(n):
                out[layer, start + t] = pools[layer][int(block_table[b, t // block_size]), t % block_size]
    return out


# ---------------------------------------------------------------------------
# 13. sparse-prefill consumer: the kept tokens' rows of a cache tensor


def gather_rows(cache: np.ndarray, kept_idx: Sequence[int]) -> np.ndarray:
    """Rows of the kept tokens of a token-major cache tensor.

    cache: [Ly, Ntot, Hk, d] (any dtype; bf16 bit patterns pass through
    unchanged); kept_idx: packed token indices from the selection.
    Returns [Ly, len(kept_idx), Hk, d] with row i = cache[:, kept_idx[i]]
    ("SpecPrefill — Implementation Guide", §How It Works / Sparse Prefill:
    the target prefills only the kept tokens, each with its original
    position).
    """
    idx = np.asarray(kept_idx, dtype=np.int64)
    return np.asarray(cache)[:, idx]
