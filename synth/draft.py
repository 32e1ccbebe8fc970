"""Attention inputs of a random-weight draft model: the keys a draft engine
caches for the prompt and the queries of its lookahead tokens.

The pages' pipeline runs a small Qwen3.5 draft over the prompt and L
lookahead tokens and reads the post-softmax attention of the draft's
full-attention layers (llama.cpp PR "Speculative prefill", §Approach items
1-2; "SpecPrefill — Implementation Guide", §How It Works / Attention
Capture). This module builds only the inputs of that attention, never the
scoring: for each full-attention layer, the key projection of every prompt
token and the query projection of every lookahead token, each followed by
the per-head RMS normalisation of Qwen-style attention (QK-norm) and the
rotary position embedding (RoPE) at the token's position.

Readings (the pages give no weights, hidden states or layer internals):
* Weights are random (no trained draft is available): projections
  N(0, 1 / hidden), QK-norm gains 1 + 0.1 N(0, 1) per head dimension.
* The hidden state entering each full-attention layer is an independent
  seeded N(0, 1) vector per token, RMS-normalised (the layer's input norm
  with unit gain); the lookahead tokens' hidden states likewise.
* RoPE rotates the first `rotary_dim` dimensions of each head in the
  rotate-half layout with frequencies theta^(-2i / rotary_dim); the default
  rotates a quarter of head_dim 256 (partial rotary, as Qwen3-Next-style
  full-attention layers do) with theta = 10^7.
* Prompt tokens sit at positions 0 .. n-1, lookahead step l at n + l.

Everything is float32 numpy, rounded once to bf16 (nearest-even); the same
bits feed the CUDA path and the oracle.
"""

from dataclasses import dataclass
from typing import List, Sequence, Tuple

import numpy as np

from .inputs import bf16_bits_from_f32

_STREAM_W, _STREAM_H, _STREAM_Y, _STREAM_PAGES = 10, 11, 12, 13


@dataclass(frozen=True)
class DraftShape:
    hidden: int = 1024          # 0.8B-like; 2048 for the 2B-like draft
    n_layers: int = 6           # full-attention layers
    n_q_heads: int = 8
    n_kv_heads: int = 2
    head_dim: int = 256
    n_lookahead: int = 8
    rotary_dim: int = 64
    rope_theta: float = 1.0e7
    eps: float = 1.0e-6
    seed: int = 2001


DRAFT_08B = DraftShape(hidden=1024, seed=2001)
DRAFT_2B = DraftShape(hidden=2048, seed=2002)


def rms_normalize(x: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) over the last axis (float32)."""
    x = np.asarray(x, dtype=np.float32)
    ms = np.mean(np.square(x, dtype=np.float32), axis=-1, keepdims=True, dtype=np.float32)
    return (x / np.sqrt(ms + np.float32(eps))).astype(np.float32)


def rope(x: np.ndarray, positions: np.ndarray, rotary_dim: int, theta: float) -> np.ndarray:
    """Rotate-half RoPE of the first rotary_dim dims of x [..., n, H, d] at
    positions [n] (float64 angles, float32 result)."""
    half = rotary_dim // 2
    inv = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / rotary_dim)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv[None, :]          # [n, half]
    cos = np.cos(ang).astype(np.float32)[:, None, :]
    sin = np.sin(ang).astype(np.float32)[:, None, :]
    out = np.array(x, dtype=np.float32, copy=True)
    x1 = x[..., :half].astype(np.float32)
    x2 = x[..., half:rotary_dim].astype(np.float32)
    out[..., :half] = x1 * cos - x2 * sin
    out[..., half:rotary_dim] = x2 * cos + x1 * sin
    return out


def _layer_weights(shape: DraftShape, layer: int):
    rng = np.random.default_rng([shape.seed, _STREAM_W, layer])
    std = np.float32(1.0 / np.sqrt(shape.hidden))
    wk = rng.standard_normal((shape.hidden, shape.n_kv_heads * shape.head_dim), dtype=np.float32) * std
    wq = rng.standard_normal((shape.hidden, shape.n_q_heads * shape.head_dim), dtype=np.float32) * std
    gk = (1.0 + 0.1 * rng.standard_normal(shape.head_dim)).astype(np.float32)
    gq = (1.0 + 0.1 * rng.standard_normal(shape.head_dim)).astype(np.float32)
    return wk, wq, gk, gq


def attention_inputs(shape: DraftShape, lengths: Sequence[int]) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(q_bits [B, Ly, L, Hq, d], k_bits [Ly, Ntot, Hk, d], seq_off [B+1]):
    the lookahead queries and the prompts' cached keys of every
    full-attention layer, prompts packed along the token axis."""
    lengths = np.asarray(lengths, dtype=np.int64)
    seq_off = np.zeros(len(lengths) + 1, dtype=np.int32)
    seq_off[1:] = np.cumsum(lengths)
    ntot = int(seq_off[-1])
    s = shape
    k = np.empty((s.n_layers, ntot, s.n_kv_heads, s.head_dim), dtype=np.uint16)
    q = np.empty((len(lengths), s.n_layers, s.n_lookahead, s.n_q_heads, s.head_dim), dtype=np.uint16)
    for layer in range(s.n_layers):
        wk, wq, gk, gq = _layer_weights(s, layer)
        for b, n in enumerate(lengths):
            n = int(n)
            lo = int(seq_off[b])
            if n > 0:
                hrng = np.random.default_rng([s.seed, _STREAM_H, layer, b])
                h = rms_normalize(hrng.standard_normal((n, s.hidden), dtype=np.float32), s.eps)
                kk = (h @ wk).reshape(n, s.n_kv_heads, s.head_dim)
                kk = rms_normalize(kk, s.eps) * gk
                kk = rope(kk, np.arange(n), s.rotary_dim, s.rope_theta)
                k[layer, lo:lo + n] = bf16_bits_from_f32(kk)
            yrng = np.random.default_rng([s.seed, _STREAM_Y, layer, b])
            y = rms_normalize(yrng.standard_normal((s.n_lookahead, s.hidden), dtype=np.float32), s.eps)
            qq = (y @ wq).reshape(s.n_lookahead, s.n_q_heads, s.head_dim)
            qq = rms_normalize(qq, s.eps) * gq
            qq = rope(qq, n + np.arange(s.n_lookahead), s.rotary_dim, s.rope_theta)
            q[b, layer] = bf16_bits_from_f32(qq)
    return q, k, seq_off


def page_keys(k_bits: np.ndarray, seq_off: Sequence[int], block_size: int,
              seed: int = 0) -> Tuple[List[np.ndarray], np.ndarray]:
    """Block-paged per-layer pools of the dense keys, as a draft engine's
    cache holds them: every prompt's tokens in blocks of block_size rows, the
    blocks of all prompts shuffled over one pool per layer (the rows past a
    prompt's end in its last block repeat its last token). Returns the pools
    [num_blocks, block_size, Hk, d] and the block table [B, max_blocks]
    (int32; logical block j of prompt b is pool block table[b, j])."""
    seq_off = np.asarray(seq_off, dtype=np.int64)
    lengths = np.diff(seq_off)
    nblk_b = (lengths + block_size - 1) // block_size
    nblk = int(nblk_b.sum())
    perm = np.random.default_rng([seed, _STREAM_PAGES, block_size]).permutation(max(nblk, 1))[:nblk]
    table = np.zeros((len(lengths), max(1, int(nblk_b.max(initial=0)))), dtype=np.int32)
    src = np.zeros(nblk * block_size, dtype=np.int64)
    first = 0
    for b, (n, nb) in enumerate(zip(lengths, nblk_b)):
        nb = int(nb)
        table[b, :nb] = perm[first:first + nb]
        for j in range(nb):
            t = np.minimum(np.arange(j * block_size, (j + 1) * block_size), int(n) - 1)
            p = int(perm[first + j])
            src[p * block_size:(p + 1) * block_size] = seq_off[b] + t
        first += nb
    ly, _, hk, d = k_bits.shape
    pools = [np.ascontiguousarray(k_bits[l][src].reshape(nblk, block_size, hk, d)) for l in range(ly)]
    return pools, table
