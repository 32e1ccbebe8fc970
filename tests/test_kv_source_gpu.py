"""GPU checks of the in-situ key sources: keys read in place from one pool
per layer (packed rows, head-major rows, or block-paged through a block
table with shuffled blocks). The same keys give the same scores and lists
as the dense [Ly][Ntot][Hk][d] path bit for bit (the tiles, and so the
arithmetic, are identical), which the dense parity tests tie to the oracle;
one case is also compared with the oracle's own gather of the pages."""

import numpy as np
import pytest

import oracle
from tests import gpu_helpers as gh
from tests._cases import random_case
from tests.test_oracle_pins import _scatter_pages
from tests.test_parity_gpu import BASE, _check_scores, _check_t1, _check_t2

pytestmark = pytest.mark.gpu

KEYS = ("imp", "tok_score", "chunk_score", "chunk_keep", "kept_idx", "kept_pos", "kept_off")


def _dense(sp, q, k, off, kw):
    import torch
    qd, kd, od = gh.to_device(type("I", (), {"q": q, "k": k, "seq_off": off})())
    out = gh.out_to_numpy(sp.specprefill_score(qd, kd, od, sp.SelectionParams(**kw)))
    torch.cuda.synchronize()
    return out, qd, od


def _kv(sp, qd, od, layer_k, ntot, kw, table=None):
    import torch
    p = sp.SelectionParams(**kw)
    shape = sp.shape_of_kv(qd, layer_k, ntot, table)
    ws = sp.make_workspace(shape, p, poison=True)
    out = sp.specprefill_score_kv(qd, layer_k, od, ntot, p, block_table=table, ws=ws)
    torch.cuda.synchronize()
    return gh.out_to_numpy(out), sp.device_status(ws)


def _bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _same(a, b):
    for key in KEYS:
        assert np.array_equal(a[key], b[key]), key


CASE = ([3000, 0, 1, 1700], 2, 8, 2, 128, 4)   # ragged, an empty and a one-token prompt


def test_per_layer_pools_equal_the_dense_path(cuda_lib):
    sp = cuda_lib
    lengths, ly, hq, hk, d, steps = CASE
    q, k, off = random_case(70, lengths, ly, hq, hk, d, steps, q_gain=2.0)
    kw = dict(BASE, mode="mass", mass=0.85)
    ref, qd, od = _dense(sp, q, k, off, kw)
    ntot = int(off[-1])
    # separate allocations, token-major rows
    pools = [_bf16(k[layer]).clone() for layer in range(ly)]
    got, st = _kv(sp, qd, od, pools, ntot, kw)
    assert st == 0
    _same(got, ref)
    # head-major rows ([Hk][rows][d] per layer, as a transposed view)
    hm = [_bf16(np.ascontiguousarray(k[layer].transpose(1, 0, 2))).transpose(0, 1) for layer in range(ly)]
    assert hm[0].stride(0) == d and hm[0].stride(1) == ntot * d
    got, st = _kv(sp, qd, od, hm, ntot, kw)
    assert st == 0
    _same(got, ref)


@pytest.mark.parametrize("bs", [8, 16, 64, 128, 256])
def test_block_paged_pools_equal_the_dense_path(cuda_lib, bs):
    import torch
    sp = cuda_lib
    lengths, ly, hq, hk, d, steps = CASE
    q, k, off = random_case(71, lengths, ly, hq, hk, d, steps, q_gain=2.0)
    kw = dict(BASE, mode="fixed", keep_p=0.25)
    ref, qd, od = _dense(sp, q, k, off, kw)
    pools, table = _scatter_pages(k, off, bs, np.random.default_rng(bs))
    dev_pools = [_bf16(pl) for pl in pools]
    got, st = _kv(sp, qd, od, dev_pools, int(off[-1]), kw, torch.from_numpy(table).cuda())
    assert st == 0
    _same(got, ref)


def test_block_paged_against_the_oracle(cuda_lib):
    """The oracle gathers the pages itself; the GPU reads them in place."""
    import torch
    sp = cuda_lib
    q, k, off = random_case(72, [2500, 900], 2, 8, 2, 256, 8, q_gain=2.0)
    pools, table = _scatter_pages(k, off, 16, np.random.default_rng(5))
    kw = dict(BASE, mode="mass", mass=0.85)
    qd, _, od = gh.to_device(type("I", (), {"q": q, "k": k, "seq_off": off})())
    got, st = _kv(sp, qd, od, [_bf16(pl) for pl in pools], int(off[-1]), kw,
                  torch.from_numpy(table).cuda())
    assert st == 0
    dense = oracle.kv_from_pages(pools, table, off, 16)
    ref = oracle.run(q, dense, off, **kw)
    _check_scores(got, ref)
    _check_t1(got, off, kw)
    _check_t2(got, ref, off, kw)


def test_bad_block_tables_are_reported(cuda_lib):
    """A block id outside the pool and a table row too short for its prompt
    both end in SP_ERR_DEVICE on the workspace, with no access outside the
    pool or the table."""
    import torch
    sp = cuda_lib
    q, k, off = random_case(73, [700, 300], 1, 4, 2, 64, 2, q_gain=2.0)
    pools, table = _scatter_pages(k, off, 16, np.random.default_rng(1))
    dev_pools = [_bf16(pl) for pl in pools]
    qd, _, od = gh.to_device(type("I", (), {"q": q, "k": k, "seq_off": off})())
    kw = dict(BASE, mode="fixed", keep_p=0.3)
    bad = table.copy()
    bad[0, 3] = 1 << 20
    bad[1, 1] = -7
    _, st = _kv(sp, qd, od, dev_pools, int(off[-1]), kw, torch.from_numpy(bad).cuda())
    assert st == 6
    short = np.ascontiguousarray(table[:, :20])     # prompt 0 needs 44 blocks
    _, st = _kv(sp, qd, od, dev_pools, int(off[-1]), kw, torch.from_numpy(short).cuda())
    assert st == 6
    # a valid call afterwards succeeds (the context is intact)
    got, st = _kv(sp, qd, od, dev_pools, int(off[-1]), kw, torch.from_numpy(table).cuda())
    assert st == 0
