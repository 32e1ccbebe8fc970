"""Seeded synthetic query/key inputs (bf16 bit patterns) for the scoring path.

Recipe (one reading of the pages' workloads, which use real drafts and
NIAH/RULER-style prompts that are not available here):

* Q and K background entries are i.i.d. N(0, 1) float32 samples, rounded to
  bf16 with round-to-nearest-even; the identical bits feed every consumer.
* A *needle* at token t for query head h replaces the key of KV head h // G
  in every layer l with 4 * RMSnorm(sum_s q[l, s, h, :]) (unit-RMS scaling,
  matching the unit-RMS background keys), so that head's lookahead queries
  attend sharply to it.  The "aligned" layout (small case) uses the step-0
  query q[l, 0, h, :] instead of the sum over steps.
* Long-context prompts add a slowly varying shift c(t) * sqrt(d) * v[l, g]
  to every key (v a random unit vector per layer/KV head, c piecewise linear
  between values drawn U(-1, 1) at region centres every 4096 tokens), which
  spreads attention over broad regions (diffuse attention).
* Re-draws for score-margin enforcement (``prompt_attempts``) change a
  prompt's queries and its needle sites (positions and heads); the key
  background is a function of the seed alone.

Random streams are numpy ``default_rng`` seeded with integer tuples, so each
stream (lengths, K per layer, Q per prompt/attempt, needles, shift) is
independent of the others and reproducible on any machine.
"""

from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import numpy as np

from .workloads import Workload

_STREAM_K, _STREAM_Q, _STREAM_NEEDLE, _STREAM_LEN, _STREAM_SHIFT = 0, 1, 2, 3, 4
REGION = 4096
NEEDLE_GAIN = 4.0


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """Exact float32 value of bf16 bit patterns."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Inputs:
    q: np.ndarray          # uint16 [B, Ly, L, Hq, d]
    k: np.ndarray          # uint16 [Ly, Ntot, Hk, d]
    seq_off: np.ndarray    # int32 [B + 1]
    needles: List[Tuple[int, int, int]]  # (prompt, token-in-prompt, query head)
    prompt_attempts: Tuple[int, ...]

    @property
    def lengths(self) -> np.ndarray:
        return np.diff(self.seq_off)

    @property
    def n_tokens_total(self) -> int:
        return int(self.seq_off[-1])


def prompt_lengths(w: Workload) -> np.ndarray:
    if w.lengths is not None:
        return np.asarray(w.lengths, dtype=np.int64)
    lo, hi = w.len_range
    rng = np.random.default_rng([w.seed, _STREAM_LEN])
    return rng.integers(lo, hi + 1, size=w.n_prompts).astype(np.int64)


def background_keys(w: Workload, lengths: Sequence[int]) -> np.ndarray:
    """Key background (with the diffuse shift when the workload has one)."""
    lengths = np.asarray(lengths, dtype=np.int64)
    n_tot = int(lengths.sum())
    hk, d = w.n_kv_heads, w.head_dim
    k = np.empty((w.n_layers, n_tot, hk, d), dtype=np.uint16)
    shift_c = shift_v = None
    if w.diffuse_shift:
        srng = np.random.default_rng([w.seed, _STREAM_SHIFT])
        v = srng.standard_normal((w.n_layers, hk, d))
        shift_v = (v / np.linalg.norm(v, axis=-1, keepdims=True)) * np.sqrt(d)
        shift_c = np.empty(n_tot, dtype=np.float64)
        start = 0
        for n in lengths:
            n = int(n)
            n_reg = (n + REGION - 1) // REGION
            centres = REGION * np.arange(n_reg) + REGION / 2.0
            values = srng.uniform(-1.0, 1.0, size=n_reg)
            shift_c[start:start + n] = np.interp(np.arange(n), centres, values)
            start += n
    for layer in range(w.n_layers):
        krng = np.random.default_rng([w.seed, _STREAM_K, layer])
        x = krng.standard_normal((n_tot, hk, d), dtype=np.float32)
        if shift_c is not None:
            x += (shift_c[:, None, None] * shift_v[layer][None, :, :]).astype(np.float32)
        k[layer] = bf16_bits_from_f32(x)
    return k


def prompt_queries(w: Workload, prompt: int, attempt: int) -> np.ndarray:
    """bf16 bits [Ly, L, Hq, d] for one prompt and re-draw attempt."""
    qrng = np.random.default_rng([w.seed, _STREAM_Q, prompt, attempt])
    x = qrng.standard_normal((w.n_layers, w.n_lookahead, w.n_q_heads, w.head_dim), dtype=np.float32)
    return bf16_bits_from_f32(x)


def needle_sites(w: Workload, prompt: int, n: int, attempt: int = 0) -> List[Tuple[int, int]]:
    """(token, query head) pairs for one prompt; tokens distinct, in [1, n-1)."""
    m = w.needles_per_prompt
    if m == 0 or n < 3:
        return []
    nrng = np.random.default_rng([w.seed, _STREAM_NEEDLE, prompt, attempt])
    if w.needle_layout in ("uniform", "aligned"):
        m = min(m, n - 2)
        toks = nrng.choice(np.arange(1, n - 1), size=m, replace=False)
    elif w.needle_layout == "clustered":
        n_sec = 8
        per = (m + n_sec - 1) // n_sec
        lo, hi = w.chunk, max(w.chunk + 1, n - w.chunk)
        centres = nrng.integers(lo, hi, size=n_sec)
        chosen: List[int] = []
        seen = set()
        for c in centres:
            got = 0
            while got < per and len(chosen) < m:
                t = int(np.clip(c + nrng.integers(-256, 257), 1, n - 2))
                if t not in seen:
                    seen.add(t)
                    chosen.append(t)
                    got += 1
        toks = np.asarray(chosen, dtype=np.int64)
    else:
        raise ValueError(w.needle_layout)
    heads = nrng.integers(0, w.n_q_heads, size=len(toks))
    return [(int(t), int(h)) for t, h in zip(toks, heads)]


def plant_needles(w: Workload, k: np.ndarray, q: np.ndarray, seq_off: np.ndarray,
                  needles: List[Tuple[int, int, int]]) -> None:
    """Overwrite needle keys in place (k: [Ly, Ntot, Hk, d] bits)."""
    g = w.group
    for (b, t, h) in needles:
        qb = f32_from_bf16_bits(q[b])  # [Ly, L, Hq, d]
        for layer in range(w.n_layers):
            if w.needle_layout == "aligned":
                v = qb[layer, 0, h, :].astype(np.float32)
            else:
                v = qb[layer, :, h, :].sum(axis=0, dtype=np.float32)
            rms = np.sqrt(np.mean(v.astype(np.float64) ** 2))
            key = (NEEDLE_GAIN * v / rms).astype(np.float32)
            k[layer, int(seq_off[b]) + t, h // g, :] = bf16_bits_from_f32(key)


def make_inputs(w: Workload, prompt_attempts: Optional[Sequence[int]] = None,
                k_background: Optional[np.ndarray] = None) -> Inputs:
    """Build one seeded input set for workload ``w``.

    ``prompt_attempts[b]`` selects prompt b's query re-draw (default 0).
    ``k_background`` may pass a cached ``background_keys`` result; it is
    copied, never modified.
    """
    lengths = prompt_lengths(w)
    b_count = len(lengths)
    if prompt_attempts is None:
        prompt_attempts = (0,) * b_count
    prompt_attempts = tuple(int(a) for a in prompt_attempts)
    assert len(prompt_attempts) == b_count
    seq_off = np.zeros(b_count + 1, dtype=np.int32)
    seq_off[1:] = np.cumsum(lengths)
    if k_background is None:
        k = background_keys(w, lengths)
    else:
        k = k_background.copy()
    q = np.stack([prompt_queries(w, b, prompt_attempts[b]) for b in range(b_count)])
    needles = []
    for b in range(b_count):
        needles += [(b, t, h) for (t, h) in needle_sites(w, b, int(lengths[b]), prompt_attempts[b])]
    plant_needles(w, k, q, seq_off, needles)
    return Inputs(q=q, k=k, seq_off=seq_off, needles=needles, prompt_attempts=prompt_attempts)
