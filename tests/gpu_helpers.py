"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
library, compare with the float64 oracle."""

import json
import os

import numpy as np

from synth import get_workload, make_inputs

HERE = os.path.dirname(os.path.abspath(__file__))
# The scoring tolerance the method's specification states for importance
# scores: |gpu - oracle| <= ATOL + RTOL * |oracle|.
RTOL = 1e-3
ATOL = 1e-5


def seeds():
    with open(os.path.join(HERE, "golden", "seeds.json")) as f:
        return json.load(f)


def workload_inputs(name):
    w = get_workload(name)
    attempts = seeds()[name]["prompt_attempts"]
    return w, make_inputs(w, prompt_attempts=attempts)


def to_device(inp, dev="cuda"):
    import torch
    q = torch.from_numpy(np.ascontiguousarray(inp.q).view(np.int16)).to(dev)
    k = torch.from_numpy(np.ascontiguousarray(inp.k).view(np.int16)).to(dev)
    off = torch.from_numpy(np.ascontiguousarray(inp.seq_off, dtype=np.int32)).to(dev)
    return q, k, off


def within_tol(got, ref, rtol=RTOL, atol=ATOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    excess = np.abs(got - ref) - (atol + rtol * np.abs(ref))
    return float(excess.max()) if excess.size else -1.0


def out_to_numpy(out, n_chunks_total=None):
    n = int(out.n_kept.item())
    res = {
        "kept_idx": out.kept_idx[:n].cpu().numpy().astype(np.int64),
        "kept_pos": out.kept_pos[:n].cpu().numpy().astype(np.int64),
        "kept_off": out.kept_off.cpu().numpy().astype(np.int64),
    }
    for key in ("imp", "tok_score", "chunk_score", "chunk_off", "chunk_keep"):
        v = getattr(out, key)
        if v is not None:
            res[key] = v.cpu().numpy()
    if "chunk_off" in res:
        total = int(res["chunk_off"][-1])
        res["chunk_score"] = res["chunk_score"][:total]
        res["chunk_keep"] = res["chunk_keep"][:total]
    return res
