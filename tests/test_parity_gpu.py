"""GPU parity of the CUDA path against the float64 oracle, through the C ABI.

Scores (imp, pooled token score, chunk score) must agree within the stated
tolerance (1e-3 relative + 1e-5 absolute); integer results (chunk flags,
kept indices and positions, offsets) must agree bit for bit:
  T1  the oracle's selection steps run on the GPU's own fp32 chunk scores
      reproduce the GPU's flags and lists exactly (selection logic);
  T2  end to end, the GPU's lists equal the oracle's wherever the oracle's
      cut-off margin is safe (all committed workload seeds guarantee it).
"""

import numpy as np
import pytest

import oracle
from tests import gpu_helpers as gh
from tests._cases import random_case
from tests.golden.margins import margins_ok, prompt_margins

pytestmark = pytest.mark.gpu

SCORE_KEYS = ("imp", "tok_score", "chunk_score")
LIST_KEYS = ("chunk_keep", "kept_idx", "kept_pos", "kept_off")


def _params(sp, kw):
    return sp.SelectionParams(**kw)


def _check_t1(got, seq_off, kw):
    t1 = oracle.select_from_chunk_scores(got["chunk_score"].astype(np.float64), seq_off, **kw)
    np.testing.assert_array_equal(got["chunk_off"], t1["chunk_off"])
    for key in LIST_KEYS:
        np.testing.assert_array_equal(got[key], t1[key], err_msg=f"T1 {key}")


def _check_scores(got, ref):
    for key in SCORE_KEYS:
        ex = gh.within_tol(got[key], ref[key])
        assert ex <= 0, f"{key} outside tolerance by {ex:.3e}"


def _safe_prompts(ref, seq_off, kw):
    coff = ref["chunk_off"]
    ok = []
    for b in range(len(seq_off) - 1):
        m = prompt_margins(ref["chunk_score"][coff[b]:coff[b + 1]], kw["mode"],
                           kw.get("keep_p", 0.3), kw.get("mass", 0.85))
        ok.append(margins_ok(m))
    return ok


def _check_t2(got, ref, seq_off, kw, require_all=False):
    safe = _safe_prompts(ref, seq_off, kw)
    if require_all:
        assert all(safe), "committed seed lost its margin"
    coff = ref["chunk_off"]
    for b, s in enumerate(safe):
        if not s:
            continue
        np.testing.assert_array_equal(got["chunk_keep"][coff[b]:coff[b + 1]],
                                      ref["chunk_keep"][coff[b]:coff[b + 1]], err_msg=f"T2 flags b={b}")
        g0, g1 = got["kept_off"][b], got["kept_off"][b + 1]
        r0, r1 = ref["kept_off"][b], ref["kept_off"][b + 1]
        np.testing.assert_array_equal(got["kept_idx"][g0:g1], ref["kept_idx"][r0:r1])
        np.testing.assert_array_equal(got["kept_pos"][g0:g1], ref["kept_pos"][r0:r1])
    if all(safe):
        for key in LIST_KEYS:
            np.testing.assert_array_equal(got[key], ref[key], err_msg=f"T2 {key}")


def _run(cuda_lib, q_np, k_np, off_np, kw):
    import torch
    sp = cuda_lib
    q = torch.from_numpy(np.ascontiguousarray(q_np).view(np.int16)).cuda()
    k = torch.from_numpy(np.ascontiguousarray(k_np).view(np.int16)).cuda()
    off = torch.from_numpy(np.asarray(off_np, dtype=np.int32)).cuda()
    p = _params(sp, kw)
    # a workspace full of NaN bytes: any read of scratch nobody wrote shows up
    ws = sp.make_workspace(sp.shape_of(q, k), p, poison=True)
    out = sp.specprefill_score(q, k, off, p, ws=ws)
    torch.cuda.synchronize()
    assert sp.device_status(ws) == 0
    return gh.out_to_numpy(out), (q, k, off)


BASE = dict(pool_w=13, chunk=32, mode="mass", keep_p=0.3, mass=0.85, normalize=True,
            boost_first_mult=1.5, boost_first_n=64, boost_last_mult=1.3, boost_last_n=128,
            force_bos=True, force_last_chunk=True)

SMALL = [
    # lengths, Ly, Hq, Hk, d, L, params
    ([512], 1, 4, 2, 64, 2, dict(mode="fixed", keep_p=0.3, normalize=False,
                                  boost_first_mult=1.0, boost_last_mult=1.0)),
    ([1000, 300, 129, 5], 2, 4, 2, 64, 3, dict(mode="mass", mass=0.85)),
    ([2049, 77], 3, 8, 2, 128, 4, dict(mode="fixed", keep_p=0.15)),
    ([1500], 2, 8, 2, 256, 8, dict(mode="mass", mass=0.5)),
    ([700, 1], 2, 6, 3, 128, 5, dict(mode="fixed", keep_p=0.5, chunk=16, pool_w=7)),
    ([640, 33, 1300], 1, 16, 1, 64, 4, dict(mode="mass", mass=0.85, chunk=64)),   # R = 64 rows
    ([3000], 1, 2, 2, 256, 1, dict(mode="fixed", keep_p=0.2, pool_w=1)),           # R = 1 row
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_cases_match_oracle(cuda_lib, case):
    lengths, ly, hq, hk, d, steps, kw = SMALL[case]
    q, k, off = random_case(500 + case, lengths, ly, hq, hk, d, steps, q_gain=2.0)
    full = dict(BASE)
    full.update(kw)
    got, _ = _run(cuda_lib, q, k, off, full)
    ref = oracle.run(q, k, off, **full)
    _check_scores(got, ref)
    _check_t1(got, off, full)
    _check_t2(got, ref, off, full)


def test_simt_and_tensor_core_logits_agree(cuda_lib):
    import torch
    sp = cuda_lib
    q, k, off = random_case(77, [3000, 517], 3, 8, 2, 256, 8, q_gain=2.0)
    qd, kd, od = gh.to_device(type("I", (), {"q": q, "k": k, "seq_off": off})())
    p = sp.SelectionParams()
    a = sp.attn_importance(qd, kd, od, p).cpu().numpy()
    b = sp.attn_importance_simt(qd, kd, od, p).cpu().numpy()
    torch.cuda.synchronize()
    assert gh.within_tol(a, b, rtol=1e-4, atol=1e-7) <= 0


@pytest.fixture(scope="module")
def workload_runs(cuda_lib):
    cache = {}

    def get(name):
        if name not in cache:
            import torch
            w, inp = gh.workload_inputs(name)
            kw = w.selection_kwargs()
            got, _ = _run(cuda_lib, inp.q, inp.k, inp.seq_off, kw)
            ref = oracle.run(inp.q, inp.k, inp.seq_off, **kw)
            cache.clear()
            cache[name] = (w, inp, kw, got, ref)
            torch.cuda.empty_cache()
        return cache[name]
    return get


WORKLOADS = ["tiny", "draft08b", "draft2b", "serving", "long_fixed", "long_mass"]


@pytest.mark.parametrize("name", WORKLOADS)
def test_workload_end_to_end(workload_runs, name):
    w, inp, kw, got, ref = workload_runs(name)
    _check_scores(got, ref)
    _check_t1(got, inp.seq_off, kw)
    _check_t2(got, ref, inp.seq_off, kw, require_all=True)
    # every planted needle of a fixed-fraction workload lands in a kept chunk
    if w.mode == "fixed":
        kept = set(got["kept_idx"].tolist())
        for (b, t, h) in inp.needles:
            assert int(inp.seq_off[b]) + t in kept


def test_stage_entry_points_compose_to_the_fused_call(cuda_lib):
    import torch
    sp = cuda_lib
    w, inp = gh.workload_inputs("draft08b")
    kw = w.selection_kwargs()
    p = sp.SelectionParams(**kw)
    q, k, off = gh.to_device(inp)
    fused = gh.out_to_numpy(sp.specprefill_score(q, k, off, p))
    ntot = inp.n_tokens_total
    imp = sp.attn_importance(q, k, off, p)
    tok = torch.empty(ntot, dtype=torch.float32, device="cuda")
    _, cs, coff = sp.pool_chunk(imp, off, p, tok_score=tok)
    keep = sp.select(cs, coff, off, ntot, p)
    idx, pos, koff, nk = sp.gather_kept(keep, coff, off, ntot, p)
    torch.cuda.synchronize()
    n = int(nk.item())
    assert np.array_equal(imp.cpu().numpy(), fused["imp"])
    assert np.array_equal(tok.cpu().numpy(), fused["tok_score"])
    total = int(coff[-1].item())
    assert np.array_equal(cs[:total].cpu().numpy(), fused["chunk_score"])
    assert np.array_equal(keep[:total].cpu().numpy(), fused["chunk_keep"])
    assert np.array_equal(idx[:n].cpu().numpy(), fused["kept_idx"])
    assert np.array_equal(pos[:n].cpu().numpy(), fused["kept_pos"])
    assert np.array_equal(koff.cpu().numpy(), fused["kept_off"])


def test_two_runs_are_bitwise_identical(cuda_lib):
    sp = cuda_lib
    w, inp = gh.workload_inputs("serving")
    p = sp.SelectionParams(**w.selection_kwargs())
    q, k, off = gh.to_device(inp)
    a = gh.out_to_numpy(sp.specprefill_score(q, k, off, p))
    b = gh.out_to_numpy(sp.specprefill_score(q, k, off, p))
    for key in a:
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("kw", [
    dict(mode="mass", mass=1.0),
    dict(mode="fixed", keep_p=1.0),
    dict(mode="fixed", keep_p=1e-4, force_bos=False, force_last_chunk=False),
    dict(mode="mass", mass=1e-4, normalize=False, boost_first_mult=1.0, boost_last_mult=1.0),
])
def test_selection_extremes(cuda_lib, kw):
    q, k, off = random_case(900, [777, 64, 3], 2, 4, 2, 64, 2, q_gain=2.0)
    full = dict(BASE)
    full.update(kw)
    got, _ = _run(cuda_lib, q, k, off, full)
    ref = oracle.run(q, k, off, **full)
    _check_scores(got, ref)
    _check_t1(got, off, full)
    if kw.get("mass") == 1.0 or kw.get("keep_p") == 1.0:
        assert got["kept_off"][-1] == off[-1]   # everything kept


def test_ragged_batch_with_empty_and_tiny_prompts(cuda_lib):
    q, k, off = random_case(901, [300, 0, 1, 12, 0, 200], 2, 4, 2, 128, 3, q_gain=2.0)
    kw = dict(BASE, mode="fixed", keep_p=0.3)
    got, _ = _run(cuda_lib, q, k, off, kw)
    ref = oracle.run(q, k, off, **kw)
    _check_scores(got, ref)
    _check_t1(got, off, kw)
    # empty prompts own no chunks and keep nothing
    assert got["kept_off"][1] == got["kept_off"][2]
    assert got["kept_off"][4] == got["kept_off"][5]


@pytest.mark.parametrize("n_prompts", [40, 63, 64, 150])
def test_many_prompt_batches_locate_every_prompt(cuda_lib, n_prompts):
    """The post kernels find each tile's or slice's prompt with a warp ballot
    over the offset tables for batches of fewer than 64 prompts and with a
    binary search above; empty prompts at the start, in the middle and at the
    end must get the offsets of their neighbours and keep nothing."""
    rng = np.random.default_rng(960 + n_prompts)
    lengths = rng.integers(1, 400, n_prompts)
    lengths[[0, n_prompts // 2, n_prompts // 2 + 1, n_prompts - 2, n_prompts - 1]] = 0
    lengths[3] = 1
    q, k, off = random_case(970 + n_prompts, lengths.tolist(), 1, 4, 2, 64, 2, q_gain=2.0)
    kw = dict(BASE, mode="fixed", keep_p=0.3)
    got, _ = _run(cuda_lib, q, k, off, kw)
    ref = oracle.run(q, k, off, **kw)
    _check_scores(got, ref)
    _check_t1(got, off, kw)
    _check_t2(got, ref, off, kw)
    for b in np.flatnonzero(lengths == 0):
        assert got["kept_off"][b] == got["kept_off"][b + 1], b


def test_invalid_offsets_set_device_status(cuda_lib):
    import torch
    sp = cuda_lib
    q, k, off = random_case(902, [200, 100], 1, 2, 1, 64, 1)
    qd, kd, _ = gh.to_device(type("I", (), {"q": q, "k": k, "seq_off": off})())
    bad = torch.tensor([0, 250, 120], dtype=torch.int32, device="cuda")  # decreasing
    p = sp.SelectionParams()
    shape = sp.shape_of(qd, kd)
    ws = sp.make_workspace(shape, p)
    sp.specprefill_score(qd, kd, bad, p, ws=ws)
    assert sp.device_status(ws) == 6
    out = sp.specprefill_score(qd, kd, torch.from_numpy(off).cuda(), p, ws=ws)
    assert sp.device_status(ws) == 0
    assert int(out.n_kept.item()) > 0


def test_max_seq_len_bound_is_checked_on_the_device(cuda_lib):
    """sp_shape.max_seq_len > 0 bounds every prompt's length: a batch with a
    longer prompt ends in SP_ERR_DEVICE, the same batch with the bound at its
    longest prompt (or no bound) is scored exactly as without it."""
    import torch
    sp = cuda_lib
    q, k, off = random_case(904, [300, 700, 64], 1, 4, 2, 64, 2, q_gain=2.0)
    qd, kd, od = gh.to_device(type("I", (), {"q": q, "k": k, "seq_off": off})())
    p = sp.SelectionParams(**dict(BASE, mode="fixed", keep_p=0.3))
    ws = sp.make_workspace(sp.shape_of(qd, kd), p)
    sp.specprefill_score(qd, kd, od, p, ws=ws, max_seq_len=699)
    assert sp.device_status(ws) == 6
    got = gh.out_to_numpy(sp.specprefill_score(qd, kd, od, p, ws=ws, max_seq_len=700))
    assert sp.device_status(ws) == 0
    free = gh.out_to_numpy(sp.specprefill_score(qd, kd, od, p, ws=ws))
    assert sp.device_status(ws) == 0
    for key in free:
        assert np.array_equal(got[key], free[key]), key
    # one prompt: the post kernels take its offsets from the token count
    q1, k1, off1 = random_case(905, [900], 1, 4, 2, 64, 2, q_gain=2.0)
    qd, kd, od = gh.to_device(type("I", (), {"q": q1, "k": k1, "seq_off": off1})())
    ws = sp.make_workspace(sp.shape_of(qd, kd), p)
    sp.specprefill_score(qd, kd, od, p, ws=ws, max_seq_len=512)
    assert sp.device_status(ws) == 6
    sp.specprefill_score(qd, kd, od, p, ws=ws, max_seq_len=900)
    assert sp.device_status(ws) == 0


@pytest.mark.parametrize("n", [1, 5, 33, 127, 128, 129, 4095])
def test_single_prompt_edge_lengths(cuda_lib, n):
    """One prompt: every kernel after the prep takes its offsets from the
    token count; lengths around the tile (128), chunk (32) and slice (1,024
    tokens) edges must match the oracle like a batch does."""
    q, k, off = random_case(1100 + n, [n], 2, 4, 2, 64, 2, q_gain=2.0)
    kw = dict(BASE, mode="fixed", keep_p=0.3)
    got, _ = _run(cuda_lib, q, k, off, kw)
    ref = oracle.run(q, k, off, **kw)
    _check_scores(got, ref)
    _check_t1(got, off, kw)
    _check_t2(got, ref, off, kw)
    assert got["kept_off"][0] == 0 and got["kept_off"][1] == len(got["kept_idx"])


def test_invalid_single_prompt_offsets_set_device_status(cuda_lib):
    """With one prompt the kernels after the prep take every offset from
    n_tokens_total and request their data before reading the prep kernel's
    decision: offsets that do not span [0, Ntot) must still end in
    SP_ERR_DEVICE, and the next valid call on the same workspace must equal
    a call on a fresh one."""
    import torch
    sp = cuda_lib
    q, k, off = random_case(903, [300], 2, 4, 2, 64, 2, q_gain=2.0)
    qd, kd, _ = gh.to_device(type("I", (), {"q": q, "k": k, "seq_off": off})())
    p = sp.SelectionParams(**dict(BASE, mode="fixed", keep_p=0.3))
    shape = sp.shape_of(qd, kd)
    ws = sp.make_workspace(shape, p, poison=True)
    for bad in ([0, 290], [5, 300], [0, 100000], [-1, 300]):
        sp.specprefill_score(qd, kd, torch.tensor(bad, dtype=torch.int32, device="cuda"), p, ws=ws)
        assert sp.device_status(ws) == 6, bad
    od = torch.from_numpy(off).cuda()
    got = gh.out_to_numpy(sp.specprefill_score(qd, kd, od, p, ws=ws))
    assert sp.device_status(ws) == 0
    fresh = gh.out_to_numpy(sp.specprefill_score(qd, kd, od, p))
    for key in fresh:
        assert np.array_equal(got[key], fresh[key]), key


def test_bounded_wait_timeout_is_reported_and_recoverable(cuda_lib):
    """A poll limit of 1 makes the first wait on a copy still in flight give
    up: the kernel records SP_ERR_TIMEOUT, drains its copies and MMAs,
    frees tensor memory and returns; the next normal call is exact."""
    import torch
    sp = cuda_lib
    w, inp = gh.workload_inputs("tiny")
    kw = w.selection_kwargs()
    q, k, off = gh.to_device(inp)
    p_fast = sp.SelectionParams(**kw, spin_limit=1)
    shape = sp.shape_of(q, k)
    ws = sp.make_workspace(shape, p_fast)
    sp.specprefill_score(q, k, off, p_fast, ws=ws)
    assert sp.device_status(ws) == 5
    p = sp.SelectionParams(**kw)
    got = gh.out_to_numpy(sp.specprefill_score(q, k, off, p, ws=ws))
    assert sp.device_status(ws) == 0
    ref = oracle.run(inp.q, inp.k, inp.seq_off, **kw)
    assert np.array_equal(got["kept_idx"], ref["kept_idx"])
