"""GPU parity of the per-head pooling variant (every attention row pooled
before the max over heads and layers) against the oracle, through the C ABI,
with the same tolerance and T1/T2 tiers as the default path."""

import numpy as np
import pytest

import oracle
from tests import gpu_helpers as gh
from tests._cases import random_case
from tests.test_parity_gpu import BASE, _check_scores, _check_t1, _check_t2, _run

pytestmark = pytest.mark.gpu

CASES = [
    # lengths, Ly, Hq, Hk, d, L, selection
    ([3000], 2, 8, 2, 128, 4, dict(mode="fixed", keep_p=0.2)),
    ([1000, 300, 129, 5, 0, 1], 2, 4, 2, 64, 3, dict(mode="mass", mass=0.85)),       # ragged, tiny, empty
    ([1500, 700], 1, 8, 2, 256, 8, dict(mode="fixed", keep_p=0.3, pool_w=129)),       # widest halo
    ([2049, 77], 3, 6, 3, 128, 5, dict(mode="mass", mass=0.6, pool_w=7, chunk=16)),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_head_pooling_matches_oracle(cuda_lib, case):
    lengths, ly, hq, hk, d, steps, sel = CASES[case]
    kw = dict(BASE, pool_at="head")
    kw.update(sel)
    q, k, off = random_case(620 + case, lengths, ly, hq, hk, d, steps, q_gain=2.0)
    got, _ = _run(cuda_lib, q, k, off, kw)
    ref = oracle.run(q, k, off, **kw)
    _check_scores(got, ref)
    np.testing.assert_array_equal(got["tok_score"], got["imp"])   # no second pooling
    _check_t1(got, off, kw)
    _check_t2(got, ref, off, kw)


def test_head_pooling_two_waves_and_64_rows(cuda_lib):
    """64 query rows per slab (L = 16, G = 4) and 16 slabs of 65K tokens
    with an 80 MiB wave budget: the scratch takes two waves, so the
    per-token maxima of the first wave are carried to the second."""
    sp = cuda_lib
    lengths = [40000, 25536]
    q, k, off = random_case(643, lengths, 4, 16, 4, 64, 16, q_gain=2.0)
    kw = dict(BASE, pool_at="head", mode="fixed", keep_p=0.25)
    got, (qd, kd, _) = _run(cuda_lib, q, k, off, dict(kw, wave_mib=80))
    assert sp.kernels_per_call(sp.shape_of(qd, kd), sp.SelectionParams(**kw, wave_mib=80)) == 8   # 2 waves
    ref = oracle.run(q, k, off, **kw)
    _check_scores(got, ref)
    _check_t1(got, off, kw)
    _check_t2(got, ref, off, kw, require_all=True)   # this seed's cut-offs have safe margins


def test_head_pooling_width_one_is_the_default_path(cuda_lib):
    q, k, off = random_case(650, [2500, 400], 2, 8, 2, 128, 4, q_gain=2.0)
    kw = dict(BASE, mode="fixed", keep_p=0.3, pool_w=1)
    a, _ = _run(cuda_lib, q, k, off, kw)
    b, _ = _run(cuda_lib, q, k, off, dict(kw, pool_at="head"))
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_head_pooling_stage_entry_points_compose(cuda_lib):
    """sp_attn_importance (pooled rows) then sp_pool_chunk, sp_select and
    sp_gather_kept with the same parameters equal the fused call."""
    import torch
    sp = cuda_lib
    q, k, off = random_case(660, [2600, 900], 2, 8, 2, 128, 4, q_gain=2.0)
    qd, kd, od = gh.to_device(type("I", (), {"q": q, "k": k, "seq_off": off})())
    p = sp.SelectionParams(**dict(BASE, pool_at="head", mode="mass", mass=0.85))
    fused = gh.out_to_numpy(sp.specprefill_score(qd, kd, od, p))
    ntot = int(off[-1])
    imp = sp.attn_importance(qd, kd, od, p)
    tok = torch.empty(ntot, dtype=torch.float32, device="cuda")
    _, cs, coff = sp.pool_chunk(imp, od, p, tok_score=tok)
    keep = sp.select(cs, coff, od, ntot, p)
    idx, pos, koff, nk = sp.gather_kept(keep, coff, od, ntot, p)
    torch.cuda.synchronize()
    n = int(nk.item())
    assert np.array_equal(imp.cpu().numpy(), fused["imp"])
    assert np.array_equal(tok.cpu().numpy(), fused["tok_score"])
    assert np.array_equal(idx[:n].cpu().numpy(), fused["kept_idx"])
    assert np.array_equal(koff.cpu().numpy(), fused["kept_off"])
