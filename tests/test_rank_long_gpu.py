"""GPU checks of the fused rank kernel on prompts of thousands of chunks.

The rank kernel decides each chunk of a slice by its position in the order
(score descending, chunk index ascending) against every chunk of its
prompt. Prompts of 2,000+ chunks beside a short one, and a prompt whose
keys are all identical, so that every token is equally important and
almost all chunk scores tie exactly, must give the oracle's selection on
the GPU's own chunk scores bit for bit (T1), scores within tolerance, and
lists end to end where the oracle's margin holds (T2). Ties are cut in
chunk order (fixed mode: by count, mass mode: by the running mass); the
listing rule keeps every chunk tied with the k-th score.
"""

import numpy as np
import pytest

import oracle
from tests._cases import random_case
from tests.test_parity_gpu import BASE, _check_scores, _check_t1, _check_t2, _run

pytestmark = pytest.mark.gpu

# small attention shape: the cost is in the token count
SHAPE = dict(n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=64, n_lookahead=2)


def _case(seed, lengths):
    return random_case(seed, lengths, SHAPE["n_layers"], SHAPE["n_q_heads"], SHAPE["n_kv_heads"],
                       SHAPE["head_dim"], SHAPE["n_lookahead"], q_gain=2.0)


LISTING = dict(rule="listing", min_tok=128, max_keep=0)


@pytest.mark.parametrize("kw", [
    dict(mode="fixed", keep_p=0.3),
    dict(mode="mass", mass=0.85),
    dict(mode="fixed", keep_p=0.1, normalize=False, boost_first_mult=1.0, boost_last_mult=1.0),
    dict(mode="fixed", keep_p=0.2, **LISTING),
])
def test_long_prompts_match_oracle(cuda_lib, kw):
    # 2,188 and 2,110 chunks beside a 94-chunk prompt
    q, k, off = _case(1300, [70000, 3000, 67500])
    full = dict(BASE, **kw)
    got, _ = _run(cuda_lib, q, k, off, full)
    ref = oracle.run(q, k, off, **full)
    _check_scores(got, ref)
    _check_t1(got, off, full)
    if kw.get("rule") != "listing":   # the listing's lists: T1 above covers them
        _check_t2(got, ref, off, full)


@pytest.mark.parametrize("kw", [
    dict(mode="fixed", keep_p=0.3),
    dict(mode="fixed", keep_p=0.05, force_bos=False, force_last_chunk=False),
    dict(mode="mass", mass=0.85),
    dict(mode="mass", mass=0.4),
    dict(mode="fixed", keep_p=0.3, **LISTING),
])
def test_tied_chunk_scores_are_cut_in_chunk_order(cuda_lib, kw):
    q, k, off = _case(1301, [66000])
    k[:] = k[:, :1]  # one key for every token: uniform attention, tied chunk scores
    # without the min-max normalisation: a constant score vector normalises
    # through max - min = 0 in fp32 and to rounding noise in float64
    full = dict(BASE, normalize=False, **kw)
    got, _ = _run(cuda_lib, q, k, off, full)
    cs = got["chunk_score"]
    assert cs.size > 2048 and np.unique(cs).size < 16   # thousands of chunks, mostly tied
    ref = oracle.run(q, k, off, **full)
    _check_scores(got, ref)
    _check_t1(got, off, full)
    keep = got["chunk_keep"] & 1
    tied = np.flatnonzero(cs == np.median(cs))
    kept_tied = tied[keep[tied] == 1]
    if kw.get("rule") == "listing":
        # the listing keeps every chunk tied with the k-th score
        assert kept_tied.size in (0, tied.size)
    else:
        # the exact rule keeps a prefix of the tied block in chunk order
        assert np.array_equal(kept_tied, tied[:kept_tied.size])
