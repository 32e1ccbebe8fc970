"""Concurrent calls and graph capture, through the C ABI.

Calls on different streams, each with its own workspace and outputs, run
concurrently (the bench's pipelined figure relies on it) and must give each
call's results bit for bit as when it runs alone. A call captured into a
CUDA graph (the library allocates nothing and synchronises nothing inside a
call) must replay to the same bits as the eager call, also after the
captured inputs have been overwritten in place with another batch.
"""

import numpy as np
import pytest

from tests import gpu_helpers as gh
from tests._cases import random_case
from tests.test_parity_gpu import BASE

pytestmark = pytest.mark.gpu

KEYS = ("imp", "tok_score", "chunk_score", "chunk_keep", "kept_idx", "kept_pos", "kept_off")


def _inputs(seed, lengths=(3000, 1200, 517), ly=2, hq=8, hk=2, d=128, steps=8):
    import torch
    q, k, off = random_case(seed, list(lengths), ly, hq, hk, d, steps, q_gain=2.0)
    return (torch.from_numpy(np.ascontiguousarray(q).view(np.int16)).cuda(),
            torch.from_numpy(np.ascontiguousarray(k).view(np.int16)).cuda(),
            torch.from_numpy(np.asarray(off, dtype=np.int32)).cuda())


def _same(a, b):
    for key in KEYS:
        x, y = np.asarray(a[key]), np.asarray(b[key])
        assert x.shape == y.shape and np.array_equal(x.view(np.uint8), y.view(np.uint8)), key


def test_concurrent_calls_on_three_streams_match_calls_alone(cuda_lib):
    import torch
    sp = cuda_lib
    p = sp.SelectionParams(**dict(BASE, mode="fixed", keep_p=0.2))
    batches = [_inputs(2100 + i) for i in range(3)]
    alone = []
    for q, k, off in batches:
        alone.append(gh.out_to_numpy(sp.specprefill_score(q, k, off, p)))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in batches]
    wss = [sp.make_workspace(sp.shape_of(q, k), p) for q, k, _ in batches]
    outs = [sp.alloc_outputs(q, k, p) for q, k, _ in batches]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for rep in range(4):   # several rounds in flight at once
        for (q, k, off), st, ws, out in zip(batches, streams, wss, outs):
            sp.specprefill_score(q, k, off, p, out=out, ws=ws, stream=st)
    torch.cuda.synchronize()
    for out, ws, ref in zip(outs, wss, alone):
        assert sp.device_status(ws) == 0
        _same(gh.out_to_numpy(out), ref)


def test_graph_captured_call_replays_bit_for_bit(cuda_lib):
    import torch
    sp = cuda_lib
    p = sp.SelectionParams(**dict(BASE, mode="mass", mass=0.85))
    q, k, off = _inputs(2200)
    q2, k2, _ = _inputs(2201)
    ws = sp.make_workspace(sp.shape_of(q, k), p)
    out = sp.alloc_outputs(q, k, p)
    eager = gh.out_to_numpy(sp.specprefill_score(q, k, off, p))
    eager2 = gh.out_to_numpy(sp.specprefill_score(q2, k2, off, p))
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        sp.specprefill_score(q, k, off, p, out=out, ws=ws, stream=st)   # warm-up outside capture
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        sp.specprefill_score(q, k, off, p, out=out, ws=ws, stream=st)
    g.replay()
    torch.cuda.synchronize()
    assert sp.device_status(ws) == 0
    _same(gh.out_to_numpy(out), eager)
    # the graph reads its inputs in place: new data, same buffers
    q.copy_(q2)
    k.copy_(k2)
    g.replay()
    torch.cuda.synchronize()
    assert sp.device_status(ws) == 0
    _same(gh.out_to_numpy(out), eager2)
