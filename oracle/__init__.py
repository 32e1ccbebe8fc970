"""Float64 CPU oracle of the SpecPrefill scoring path — TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import anything here. The CUDA library and its Python binding never
do, and share no code with it. Parity of the whole oracle is pinned by the
``-m "not gpu"`` tests (brute-force twin, closed forms, library routines and
invariants); no function here is left unpinned.
"""

from .specprefill_oracle import (  # noqa: F401
    attention_rows,
    auto_window,
    avg_pool,
    chunk_means,
    chunk_offsets,
    decode_bf16,
    finish_selection,
    gather_rows,
    fixed_count,
    importance,
    kv_from_pages,
    listing_cap,
    listing_eff_min,
    listing_forced_tokens,
    listing_keep_count,
    merge_windows,
    min_max_normalize,
    pool_rows,
    rank_order,
    run,
    select_fixed,
    score_from_importance,
    select_from_chunk_scores,
    select_listing,
    select_mass,
    select_prompt,
    step_importance,
    structural_boost,
    token_importance,
    window_plan,
)
