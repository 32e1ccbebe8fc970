"""The allocation-free pool/chunk entry point, through the C ABI.

sp_pool_chunk_noalloc serves callers that cannot allocate device memory
when they call the library (a pool that owns all device memory, a plugin
without an allocator, a loop that must not risk the device synchronisation
of cudaMalloc/cudaFree). It keeps its scratch in a fixed array inside the
library, shared by every call in the context. It runs the same kernels as
sp_pool_chunk, so two calls in a row with different batches must each equal
the workspace-based entry point bit for bit (the second call must not see
anything the first one left in the shared scratch) and agree with the
oracle within the scoring tolerance. A call with invalid offsets reports
SP_ERR_DEVICE through status_out, and the next valid call reports SP_OK
again. This file sorts last so that a stop-at-first-failure run has run
everything else.
"""

import numpy as np
import pytest

import oracle
from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _batch(seed, lengths):
    import torch
    rng = np.random.default_rng(seed)
    off = np.zeros(len(lengths) + 1, dtype=np.int32)
    off[1:] = np.cumsum(lengths)
    imp = (rng.random(int(off[-1])) ** 4 * 1e-2).astype(np.float32)
    return torch.from_numpy(imp).cuda(), torch.from_numpy(off).cuda()


def _noalloc(sp, imp, off, p, n_chunks):
    import torch
    tok = torch.full_like(imp, float("nan"))
    cs = torch.full((n_chunks,), float("nan"), dtype=torch.float32, device="cuda")
    coff = torch.full((off.numel(),), -1, dtype=torch.int32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    sp.pool_chunk_noalloc(imp, off, p, tok, cs, coff, status=status)
    torch.cuda.synchronize()
    return tok, cs, coff, int(status.item())


def test_noalloc_pool_chunk_matches_workspace_entry_on_consecutive_calls(cuda_lib):
    import torch
    sp = cuda_lib
    kw = dict(pool_w=13, chunk=32, mode="mass", mass=0.85, normalize=True)
    p = sp.SelectionParams(**kw)
    for seed, lengths in ((11, [5000, 300, 4097, 1, 12000]), (12, [700, 0, 33, 2049])):
        imp, off = _batch(seed, lengths)
        ref_tok = torch.empty_like(imp)
        _, ref_cs, ref_off = sp.pool_chunk(imp, off, p, tok_score=ref_tok)
        tok, cs, coff, status = _noalloc(sp, imp, off, p, ref_cs.numel())
        assert status == 0
        assert np.array_equal(coff.cpu().numpy(), ref_off.cpu().numpy())
        n = int(ref_off[-1].item())
        # the same kernels on the same inputs: bit for bit
        assert np.array_equal(tok.cpu().numpy().view(np.uint32), ref_tok.cpu().numpy().view(np.uint32))
        assert np.array_equal(cs[:n].cpu().numpy().view(np.uint32),
                              ref_cs[:n].cpu().numpy().view(np.uint32))
        # and the oracle's pooled and chunk scores within the scoring tolerance
        ref = oracle.score_from_importance(imp.cpu().numpy(), off.cpu().numpy(), **kw)
        assert gh.within_tol(tok.cpu().numpy(), ref["tok_score"]) <= 0
        assert gh.within_tol(cs[:n].cpu().numpy(), ref["chunk_score"]) <= 0


def test_noalloc_reports_bad_offsets_then_recovers(cuda_lib):
    import torch
    sp = cuda_lib
    p = sp.SelectionParams(mode="mass")
    imp, off = _batch(13, [900, 100, 24])
    bad = off.clone()
    bad[-1] = bad[-1] - 1          # the last offset is not the token count
    n_chunks = 1024 // 32 + 3
    _, _, _, status = _noalloc(sp, imp, bad, p, n_chunks)
    assert status == 6             # SP_ERR_DEVICE
    tok, cs, coff, status = _noalloc(sp, imp, off, p, n_chunks)
    assert status == 0
    ref_tok = torch.empty_like(imp)
    _, ref_cs, ref_off = sp.pool_chunk(imp, off, p, tok_score=ref_tok)
    n = int(ref_off[-1].item())
    assert np.array_equal(tok.cpu().numpy().view(np.uint32), ref_tok.cpu().numpy().view(np.uint32))
    assert np.array_equal(cs[:n].cpu().numpy().view(np.uint32), ref_cs[:n].cpu().numpy().view(np.uint32))
