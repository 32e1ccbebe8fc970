"""Small seeded random cases shared by the oracle pins and the GPU parity tests."""

import numpy as np

from synth import bf16_bits_from_f32


def random_case(seed, lengths, n_layers, n_q_heads, n_kv_heads, head_dim, n_lookahead,
                q_gain=1.0, k_gain=1.0):
    """bf16-bit Q [B, Ly, L, Hq, d], K [Ly, Ntot, Hk, d] and seq_off [B+1]."""
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int64)
    seq_off = np.zeros(len(lengths) + 1, dtype=np.int32)
    seq_off[1:] = np.cumsum(lengths)
    q = rng.standard_normal((len(lengths), n_layers, n_lookahead, n_q_heads, head_dim),
                            dtype=np.float32) * q_gain
    k = rng.standard_normal((n_layers, int(seq_off[-1]), n_kv_heads, head_dim),
                            dtype=np.float32) * k_gain
    return bf16_bits_from_f32(q), bf16_bits_from_f32(k), seq_off
