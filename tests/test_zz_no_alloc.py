"""The allocation-free pool/chunk entry point, through the C ABI.

sp_pool_chunk_noalloc serves callers that cannot allocate device memory
when they call the library (a pool that owns all device memory, a plugin
without an allocator, a loop that must not risk the device synchronisation
of cudaMalloc/cudaFree). It keeps its scratch in a fixed array inside the
library, shared by every call on the GPU. Two calls in a row with different
batches must each match the workspace-based sp_pool_chunk: the second call
must not see anything the first one left in the shared scratch. This file
sorts last so that a stop-at-first-failure run has run everything else.
"""

import numpy as np
import pytest

from tests import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _batch(seed, lengths):
    import torch
    rng = np.random.default_rng(seed)
    off = np.zeros(len(lengths) + 1, dtype=np.int32)
    off[1:] = np.cumsum(lengths)
    imp = (rng.random(int(off[-1])) ** 4 * 1e-2).astype(np.float32)
    return torch.from_numpy(imp).cuda(), torch.from_numpy(off).cuda()


def test_noalloc_pool_chunk_matches_workspace_entry_on_consecutive_calls(cuda_lib):
    import torch
    sp = cuda_lib
    p = sp.SelectionParams(mode="mass", mass=0.85, normalize=True)
    for seed, lengths in ((11, [5000, 300, 4097, 1, 12000]), (12, [700, 0, 33, 2049])):
        imp, off = _batch(seed, lengths)
        _, ref_cs, ref_off = sp.pool_chunk(imp, off, p, tok_score=torch.empty_like(imp))
        ref_tok = torch.empty_like(imp)
        sp.pool_chunk(imp, off, p, tok_score=ref_tok)
        tok = torch.full_like(imp, float("nan"))
        cs = torch.full_like(ref_cs, float("nan"))
        coff = torch.full_like(ref_off, -1)
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        sp.pool_chunk_noalloc(imp, off, p, tok, cs, coff, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(coff.cpu().numpy(), ref_off.cpu().numpy())
        n = int(ref_off[-1].item())
        assert gh.within_tol(tok.cpu().numpy(), ref_tok.cpu().numpy()) <= 0
        assert gh.within_tol(cs[:n].cpu().numpy(), ref_cs[:n].cpu().numpy()) <= 0
