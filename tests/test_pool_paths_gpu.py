"""GPU parity of the fused post path's pooling (pool_sums_kernel: pooled
scores, tile min / max and chunk sums in one kernel per 128-token tile)
against the staged entry points (importance kernel, then the pool kernel):
imp and pooled scores equal bit for bit, and within 1e-3 relative + 1e-5
absolute of the float64 oracle, across halo widths (W = 3 .. 129), 32 and
64 query rows per slab, chunks of 16 to 128 tokens, prompts shorter than the
halo, and two waves with token pooling (the first wave's maxima carried into
the second)."""

import numpy as np
import pytest

import oracle
from tests import gpu_helpers as gh
from tests._cases import random_case
from tests.test_parity_gpu import BASE, _check_scores, _check_t1, _check_t2, _run

pytestmark = pytest.mark.gpu

CASES = [
    # lengths, Ly, Hq, Hk, d, L, params
    ([2049, 77, 1, 300], 2, 8, 2, 128, 4, dict(mode="fixed", keep_p=0.3, pool_w=129)),
    ([1000, 6, 513], 1, 16, 1, 64, 4, dict(mode="mass", mass=0.85, pool_w=13)),      # 64 rows
    ([640, 1300, 40], 3, 16, 1, 64, 4, dict(mode="fixed", keep_p=0.2, pool_w=129)),  # 64 rows, widest halo
    ([3000], 1, 2, 2, 256, 1, dict(mode="mass", mass=0.6, pool_w=3, chunk=128)),
    ([3000, 70], 1, 2, 2, 256, 1, dict(mode="mass", mass=0.6, pool_w=3, chunk=64)),
    ([257, 129, 128, 127], 2, 4, 2, 64, 2, dict(mode="fixed", keep_p=0.5, pool_w=65, chunk=16)),
]


def _staged(sp, qd, kd, od, p, ntot):
    import torch
    imp = sp.attn_importance(qd, kd, od, p)
    tok = torch.empty(ntot, dtype=torch.float32, device="cuda")
    sp.pool_chunk(imp, od, p, tok_score=tok)
    torch.cuda.synchronize()
    return imp.cpu().numpy(), tok.cpu().numpy()


@pytest.mark.parametrize("case", range(len(CASES)))
def test_fused_post_pooling_equals_the_staged_kernels(cuda_lib, case):
    sp = cuda_lib
    lengths, ly, hq, hk, d, steps, kw = CASES[case]
    q, k, off = random_case(900 + case, lengths, ly, hq, hk, d, steps, q_gain=2.0)
    full = dict(BASE, **kw)
    got, (qd, kd, od) = _run(cuda_lib, q, k, off, full)
    p = sp.SelectionParams(**full)
    assert sp.kernels_per_call(sp.shape_of(qd, kd), p) == 6   # prep, logits, importance, pool sums, rank, gather
    imp, tok = _staged(sp, qd, kd, od, p, int(off[-1]))
    assert np.array_equal(got["imp"], imp)
    assert np.array_equal(got["tok_score"], tok)
    ref = oracle.run(q, k, off, **full)
    _check_scores(got, ref)
    _check_t1(got, off, full)
    _check_t2(got, ref, off, full)


def test_token_pooling_after_a_first_wave(cuda_lib):
    """16 slabs of 64 rows over 65K tokens take two waves with an 80 MiB
    wave budget: the second wave's importance kernel combines the first
    wave's per-token maxima."""
    sp = cuda_lib
    lengths = [40000, 25536]
    q, k, off = random_case(643, lengths, 4, 16, 4, 64, 16, q_gain=2.0)
    kw = dict(BASE, mode="fixed", keep_p=0.25, pool_w=129)
    got, (qd, kd, od) = _run(cuda_lib, q, k, off, dict(kw, wave_mib=80))
    p = sp.SelectionParams(**kw, wave_mib=80)
    assert sp.kernels_per_call(sp.shape_of(qd, kd), p) == 8   # prep, 2 x (logits, importance), pool sums, rank, gather
    imp, tok = _staged(sp, qd, kd, od, p, int(off[-1]))
    assert np.array_equal(got["imp"], imp)
    assert np.array_equal(got["tok_score"], tok)
    ref = oracle.run(q, k, off, **kw)
    _check_scores(got, ref)
    _check_t1(got, off, kw)
    _check_t2(got, ref, off, kw)
