"""GPU parity of the sparse-prefill consumer gathers (kept cache rows and
kept token ids) against the oracle's gather, through the C ABI. Both are
byte copies, so the bar is bit-exact."""

import numpy as np
import pytest

import oracle
from tests import gpu_helpers as gh
from tests._cases import random_case

pytestmark = pytest.mark.gpu


def _dev_i32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _bf16(a_bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a_bits).view(np.int16)).cuda().view(torch.bfloat16)


def _bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_draft_workload_rows_follow_the_selection(cuda_lib):
    """The oracle's kept list of the 2B-draft workload gathers the same K
    rows on both sides; the GPU's own list, chained on the device from the
    scoring call, gives the same bytes."""
    import torch
    sp = cuda_lib
    w, inp = gh.workload_inputs("draft2b")
    kw = w.selection_kwargs()
    ref = oracle.run(inp.q, inp.k, inp.seq_off, **kw)
    kept = np.asarray(ref["kept_idx"], dtype=np.int64)
    want = oracle.gather_rows(inp.k, kept)
    q, k, off = gh.to_device(inp)
    kb = k.view(torch.bfloat16)
    n = len(kept)
    idx = _dev_i32(np.concatenate([kept, np.zeros(inp.n_tokens_total - n, np.int64)]))
    nk = _dev_i32([n])
    out = sp.gather_rows(kb, idx, nk)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out[:, :n]), want)
    # chained: scoring call -> gather, no host round trip in between
    res = sp.specprefill_score(q, k, off, sp.SelectionParams(**kw))
    out2 = sp.gather_rows(kb, res.kept_idx, res.n_kept)
    torch.cuda.synchronize()
    assert int(res.n_kept.item()) == n
    assert np.array_equal(_bits(out2[:, :n]), want)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_strided_cache_ragged_counts_and_spare_rows(cuda_lib, d):
    """A cache whose heads are a strided view of a wider tensor, a kept
    count below the list length, and an output with more rows than tokens:
    rows below n_kept match the oracle, the rest stay as they were."""
    import torch
    sp = cuda_lib
    ly, ntot, hk = 3, 1000 + d, 3
    _, kbits, _ = random_case(900 + d, [ntot], ly, hk, hk, d, 1)
    wide = np.zeros((ly, ntot, 2 * hk, d), np.uint16)
    wide[:, :, ::2] = kbits
    cache = _bf16(wide)[:, :, ::2]
    assert not cache.is_contiguous()
    rng = np.random.default_rng(d)
    kept = np.sort(rng.choice(ntot, size=ntot // 3, replace=False))
    n = len(kept) - 7                       # ragged: the list is longer than the count
    out = torch.full((ly, ntot + 5, hk, d), 3.0, dtype=torch.bfloat16, device="cuda")
    sentinel = _bits(out).copy()
    sp.gather_rows(cache, _dev_i32(kept), _dev_i32([n]), out=out)
    torch.cuda.synchronize()
    got = _bits(out)
    assert np.array_equal(got[:, :n], oracle.gather_rows(kbits, kept[:n]))
    assert np.array_equal(got[:, n:], sentinel[:, n:])


def test_edge_counts_and_invalid_indices(cuda_lib):
    """n_kept = 0 writes nothing; n_kept above the token count is clamped;
    an index outside the cache gives a zero row (and -1 as a token id)."""
    import torch
    sp = cuda_lib
    ly, ntot, hk, d = 2, 300, 2, 64
    _, kbits, _ = random_case(31, [ntot], ly, hk, hk, d, 1)
    cache = _bf16(kbits)
    out = torch.zeros((ly, ntot, hk, d), dtype=torch.bfloat16, device="cuda")
    perm = np.random.default_rng(5).permutation(ntot)
    sp.gather_rows(cache, _dev_i32(perm), _dev_i32([0]), out=out)
    torch.cuda.synchronize()
    assert not _bits(out).any()
    sp.gather_rows(cache, _dev_i32(perm), _dev_i32([10 * ntot]), out=out)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), oracle.gather_rows(kbits, perm))
    bad = perm.copy()
    bad[[0, 17, 299]] = [-1, ntot, 1 << 30]
    got = _bits(sp.gather_rows(cache, _dev_i32(bad), _dev_i32([ntot])))
    want = oracle.gather_rows(kbits, np.where((bad >= 0) & (bad < ntot), bad, 0))
    want[:, [0, 17, 299]] = 0
    assert np.array_equal(got, want)
    ids = np.random.default_rng(6).integers(0, 150000, size=ntot).astype(np.int32)
    tok = sp.gather_tokens(_dev_i32(ids), _dev_i32(bad), _dev_i32([ntot])).cpu().numpy()
    want_ids = oracle.gather_rows(ids[None, :], np.where((bad >= 0) & (bad < ntot), bad, 0))[0]
    want_ids[[0, 17, 299]] = -1
    assert np.array_equal(tok, want_ids)


def test_token_ids_of_a_ragged_batch(cuda_lib):
    """Kept token ids of a packed ragged batch (an empty and a one-token
    prompt among them), for the oracle's kept list of that batch."""
    import torch
    sp = cuda_lib
    lengths = [700, 0, 1, 1300]
    q, k, off = random_case(41, lengths, 2, 4, 2, 128, 3, q_gain=2.0)
    ref = oracle.run(q, k, off, pool_w=13, chunk=32, mode="mass", mass=0.85)
    ntot = int(off[-1])
    ids = np.random.default_rng(8).integers(0, 1 << 20, size=ntot).astype(np.int32)
    kept = np.asarray(ref["kept_idx"], dtype=np.int64)
    n = len(kept)
    idx = _dev_i32(np.concatenate([kept, np.full(ntot - n, -5, np.int64)]))
    tok = sp.gather_tokens(_dev_i32(ids), idx, _dev_i32([n]))
    torch.cuda.synchronize()
    assert np.array_equal(tok[:n].cpu().numpy(), oracle.gather_rows(ids[None, :], kept)[0])
