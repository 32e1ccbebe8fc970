"""GPU parity of the path's variants on the serving workload (16 prompts of
4K-16K tokens, 169K tokens in all, mass selection): the listing rule with a
2,000-token cap, per-head pooling, and keys read in place from block-paged
per-layer pools. Same bar as the default path: scores within 1e-3 relative +
1e-5 absolute of the float64 oracle, integer results bit for bit (T1 on the
GPU's own chunk scores; T2 end to end, every prompt of the committed seeds
having a safe cut-off margin)."""

import numpy as np
import pytest

import oracle
from tests import gpu_helpers as gh
from tests.test_listing_gpu import _listing_margin_ok
from tests.test_oracle_pins import _scatter_pages
from tests.test_parity_gpu import _check_scores, _check_t1, _check_t2, _run

pytestmark = pytest.mark.gpu

LIST_KEYS = ("chunk_keep", "kept_idx", "kept_pos", "kept_off")


@pytest.fixture(scope="module")
def serving():
    w, inp = gh.workload_inputs("serving")
    return w.selection_kwargs(), inp


def test_serving_listing_rule(cuda_lib, serving):
    kw0, inp = serving
    kw = dict(kw0, rule="listing", min_tok=128, max_keep=2000)
    got, _ = _run(cuda_lib, inp.q, inp.k, inp.seq_off, kw)
    ref = oracle.run(inp.q, inp.k, inp.seq_off, **kw)
    _check_scores(got, ref)
    _check_t1(got, inp.seq_off, kw)
    coff = ref["chunk_off"]
    for b in range(len(inp.seq_off) - 1):
        assert _listing_margin_ok(ref["chunk_score"][coff[b]:coff[b + 1]], kw), b
    for key in LIST_KEYS:
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    assert (np.diff(got["kept_off"]) <= 2000).all()


def test_serving_head_pooling(cuda_lib, serving):
    kw0, inp = serving
    kw = dict(kw0, pool_at="head")
    got, _ = _run(cuda_lib, inp.q, inp.k, inp.seq_off, kw)
    ref = oracle.run(inp.q, inp.k, inp.seq_off, **kw)
    _check_scores(got, ref)
    _check_t1(got, inp.seq_off, kw)
    _check_t2(got, ref, inp.seq_off, kw, require_all=True)


def test_serving_block_paged_keys_equal_the_dense_path(cuda_lib, serving):
    import torch
    sp = cuda_lib
    kw, inp = serving
    dense, _ = _run(cuda_lib, inp.q, inp.k, inp.seq_off, kw)
    pools, table = _scatter_pages(inp.k, inp.seq_off, 16, np.random.default_rng(16))
    dev_pools = [torch.from_numpy(np.ascontiguousarray(pl).view(np.int16)).cuda().view(torch.bfloat16)
                 for pl in pools]
    qd, _, od = gh.to_device(inp)
    p = sp.SelectionParams(**kw)
    ntot = int(inp.n_tokens_total)
    tbl = torch.from_numpy(table).cuda()
    ws = sp.make_workspace(sp.shape_of_kv(qd, dev_pools, ntot, tbl), p, poison=True)
    out = sp.specprefill_score_kv(qd, dev_pools, od, ntot, p, block_table=tbl, ws=ws)
    torch.cuda.synchronize()
    assert sp.device_status(ws) == 0
    got = gh.out_to_numpy(out)
    for key in ("imp", "tok_score", "chunk_score") + LIST_KEYS:
        assert np.array_equal(got[key], dense[key]), key
