"""In-situ scoring of a random-weight draft model's cache on the GPU.

The keys come from a Qwen-style draft's full-attention layers (random
weights, seeded hidden states; projection, QK-norm and RoPE, see
synth/draft.py) and sit in a cache of 16-token blocks shuffled over one pool
per layer; the queries are the draft's L lookahead tokens. The library
scores the cache in place (sp_specprefill_score_kv); the oracle scores the
dense keys it gathers from the same pages. Scores must agree within the
stated tolerance, the selection must be the oracle's on the GPU's own chunk
scores (T1) and end to end wherever the oracle's cut-off margin holds (T2),
and the paged call must equal the dense call bit for bit."""

import numpy as np
import pytest

import oracle
from synth import DraftShape, draft_attention_inputs, page_keys
from tests import gpu_helpers as gh
from tests.test_parity_gpu import BASE, _check_scores, _check_t1, _check_t2

pytestmark = pytest.mark.gpu

SHAPE = DraftShape(hidden=256, n_layers=6, n_q_heads=8, n_kv_heads=2, head_dim=256, n_lookahead=8,
                   rotary_dim=64, seed=2011)
LENGTHS = [2500, 700, 1290]
KEYS = ("imp", "tok_score", "chunk_score", "chunk_keep", "kept_idx", "kept_pos", "kept_off")


@pytest.fixture(scope="module")
def draft():
    q, k, off = draft_attention_inputs(SHAPE, LENGTHS)
    pools, table = page_keys(k, off, 16, seed=4)
    return q, k, off, pools, table


@pytest.mark.parametrize("sel", [dict(mode="fixed", keep_p=0.15), dict(mode="mass", mass=0.85)])
def test_draft_cache_scored_in_place_matches_oracle(cuda_lib, draft, sel):
    import torch
    sp = cuda_lib
    q, k, off, pools, table = draft
    kw = dict(BASE, **sel)
    p = sp.SelectionParams(**kw)
    qd = torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).cuda()
    od = torch.from_numpy(off).cuda()
    layer_k = [torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in pools]
    td = torch.from_numpy(table).cuda()
    ntot = int(off[-1])
    shape = sp.shape_of_kv(qd, layer_k, ntot, td)
    ws = sp.make_workspace(shape, p, poison=True)
    got = gh.out_to_numpy(sp.specprefill_score_kv(qd, layer_k, od, ntot, p, block_table=td, ws=ws))
    assert sp.device_status(ws) == 0
    dense = oracle.kv_from_pages(pools, table, off, 16)
    assert np.array_equal(dense, k)
    ref = oracle.run(q, dense, off, **kw)
    _check_scores(got, ref)
    _check_t1(got, off, kw)
    _check_t2(got, ref, off, kw)
    # the same keys in the dense layout: the same tiles, bit for bit
    kd = torch.from_numpy(np.ascontiguousarray(k).view(np.int16)).cuda()
    flat = gh.out_to_numpy(sp.specprefill_score(qd, kd, od, p))
    for key in KEYS:
        assert np.array_equal(got[key], flat[key]), key
