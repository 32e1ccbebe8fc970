"""Workload descriptions: shapes, needle layout and selection settings.

Shapes follow the drafts the SpecPrefill pages run: a Qwen3.5-style hybrid
model whose full-attention layers (6 in the 0.8B/2B drafts) expose KV-cached
keys, 8 query heads over 2 KV heads, head_dim 256, and 8 lookahead queries
("Speculative prefill", llama.cpp PR #27692, §Approach item 1;
"SpecPrefill — Implementation Guide", §How It Works / Attention Capture).
Selection settings follow the guide's configuration reference: W=13 pool
(PR §Approach item 3), 32-token chunks, fixed keep fraction or cumulative
mass 0.85, structural boost x1.5 on the first 64 / x1.3 on the last 128
tokens (guide v3, §v3 Improvements items 1-2, §Configuration Reference).

Plain values only; nothing here computes any part of the method.
"""

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    # prompt lengths: fixed tuple, or drawn uniformly in len_range (inclusive)
    lengths: Optional[Tuple[int, ...]]
    n_prompts: int
    len_range: Optional[Tuple[int, int]]
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_lookahead: int
    # needles
    needles_per_prompt: int
    needle_layout: str  # "aligned" | "uniform" | "clustered"
    diffuse_shift: bool
    seed: int
    # selection settings
    pool_w: int = 13
    chunk: int = 32
    mode: str = "fixed"  # "fixed" | "mass"
    keep_p: float = 0.30
    mass: float = 0.85
    normalize: bool = True
    boost_first_mult: float = 1.5
    boost_first_n: int = 64
    boost_last_mult: float = 1.3
    boost_last_n: int = 128
    force_bos: bool = True
    force_last_chunk: bool = True

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def rows_per_slab(self) -> int:
        return self.n_lookahead * self.group

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    def selection_kwargs(self) -> dict:
        """Selection settings as keyword arguments (names shared by the
        oracle and the binding; values only)."""
        return dict(
            pool_w=self.pool_w,
            chunk=self.chunk,
            mode=self.mode,
            keep_p=self.keep_p,
            mass=self.mass,
            normalize=self.normalize,
            boost_first_mult=self.boost_first_mult,
            boost_first_n=self.boost_first_n,
            boost_last_mult=self.boost_last_mult,
            boost_last_n=self.boost_last_n,
            force_bos=self.force_bos,
            force_last_chunk=self.force_last_chunk,
        )


_DRAFT = dict(n_layers=6, n_q_heads=8, n_kv_heads=2, head_dim=256, n_lookahead=8)

WORKLOADS = {
    # N=512, 1 layer, 4/2 heads, d=64, L=2, 3 needles aligned to one head's
    # step-0 query; fixed p=0.30, no normalisation, no boost.
    "tiny": Workload(
        name="tiny", lengths=(512,), n_prompts=1, len_range=None,
        n_layers=1, n_q_heads=4, n_kv_heads=2, head_dim=64, n_lookahead=2,
        needles_per_prompt=3, needle_layout="aligned", diffuse_shift=False,
        seed=1001, mode="fixed", keep_p=0.30, normalize=False,
        boost_first_mult=1.0, boost_last_mult=1.0,
    ),
    # 0.8B-draft-like: N=8192, 16 needles at random depths, mass 0.85.
    "draft08b": Workload(
        name="draft08b", lengths=(8192,), n_prompts=1, len_range=None,
        needles_per_prompt=16, needle_layout="uniform", diffuse_shift=False,
        seed=1002, mode="mass", mass=0.85, normalize=True, **_DRAFT,
    ),
    # 2B-draft-like: N=32768, 64 needles clustered in 8 sections, fixed p=0.15.
    "draft2b": Workload(
        name="draft2b", lengths=(32768,), n_prompts=1, len_range=None,
        needles_per_prompt=64, needle_layout="clustered", diffuse_shift=False,
        seed=1003, mode="fixed", keep_p=0.15, normalize=True, **_DRAFT,
    ),
    # Serving batch: 16 ragged prompts, lengths U[4096, 16384], packed.
    "serving": Workload(
        name="serving", lengths=None, n_prompts=16, len_range=(4096, 16384),
        needles_per_prompt=8, needle_layout="uniform", diffuse_shift=False,
        seed=1004, mode="mass", mass=0.85, normalize=True, **_DRAFT,
    ),
    # Long context: N=131072, 16/4 heads, d=128, diffuse shift + 32 needles.
    "long_fixed": Workload(
        name="long_fixed", lengths=(131072,), n_prompts=1, len_range=None,
        n_layers=6, n_q_heads=16, n_kv_heads=4, head_dim=128, n_lookahead=8,
        needles_per_prompt=32, needle_layout="uniform", diffuse_shift=True,
        seed=1005, mode="fixed", keep_p=0.30, normalize=True,
    ),
    "long_mass": Workload(
        name="long_mass", lengths=(131072,), n_prompts=1, len_range=None,
        n_layers=6, n_q_heads=16, n_kv_heads=4, head_dim=128, n_lookahead=8,
        needles_per_prompt=32, needle_layout="uniform", diffuse_shift=True,
        seed=1006, mode="mass", mass=0.85, normalize=True,
    ),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]
