"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports
every symbol declared in include/*.h, and rejects bad arguments on the host
(these calls enqueue nothing, so no GPU is needed)."""

import ctypes
import os
import re

import pytest

import speculative_prefill_token_gb300 as sp
from speculative_prefill_token_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sp.load()


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(sp_[a-z_0-9]+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for required in ("sp_attn_importance", "sp_pool_chunk", "sp_select", "sp_gather_kept",
                     "sp_specprefill_score", "sp_workspace_size", "sp_get_device_status"):
        assert required in names


def _comment_before(text, name):
    """The block comment directly above the declaration of `name`."""
    m = re.search(r"/\*((?:(?!\*/).)*?)\*/\s*(?:int|const char\*)\s+" + name + r"\s*\(", text, flags=re.S)
    assert m, f"no comment above {name}"
    return " ".join(m.group(1).replace("*", " ").split())


def test_each_method_entry_point_cites_its_passage():
    text = open(os.path.join(ROOT, "include", "specprefill.h")).read()
    cites = {
        "sp_attn_importance": ("Token Importance", "Attention Capture"),
        "sp_pool_chunk": ("§Approach item 3", "§Chunk Selection"),
        "sp_select": ("§Chunk Selection", "§v3 Improvements item 1", "§Approach item 4"),
        "sp_gather_kept": ("Sparse Prefill",),
        "sp_specprefill_score": ("Token Importance", "Sparse Prefill", "§Approach items 1-4"),
    }
    for name, needles in cites.items():
        comment = _comment_before(text, name)
        for needle in needles:
            assert needle in comment, f"{name}: no '{needle}' in its comment"


def test_max_seq_len_field_is_the_shape_bound(lib):
    assert [f for f, _ in sp._Shape._fields_][7] == "max_seq_len"
    s = _shape()
    s.max_seq_len = -1
    rc, _ = _ws(s, sp.SelectionParams())
    assert rc == 1
    s.max_seq_len = 4096
    rc, _ = _ws(s, sp.SelectionParams())
    assert rc == 0


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} is declared but not exported"


def test_build_info_and_status_strings(lib):
    assert b"sm_103a" in lib.sp_build_info()
    assert lib.sp_status_string(0) == b"ok"
    assert lib.sp_status_string(5) == b"a bounded device wait gave up"
    assert lib.sp_status_string(99) == b"unknown status"


def _shape(**kw):
    base = dict(n_seqs=1, n_layers=6, n_q_heads=8, n_kv_heads=2, head_dim=256, n_lookahead=8,
                n_tokens_total=32768)
    base.update(kw)
    d, ntot, hk = base["head_dim"], base["n_tokens_total"], base["n_kv_heads"]
    hq, steps, ly = base["n_q_heads"], base["n_lookahead"], base["n_layers"]
    return sp._Shape(base["n_seqs"], ly, hq, hk, d, steps, ntot, 0,
                     ntot * hk * d, hk * d, d, ly * steps * hq * d, steps * hq * d, hq * d, d)


def _ws(shape, params):
    n = ctypes.c_size_t()
    rc = sp.lib().sp_workspace_size(ctypes.byref(shape), ctypes.byref(params._c()), ctypes.byref(n))
    return rc, n.value


def test_workspace_size_valid(lib):
    rc, n = _ws(_shape(), sp.SelectionParams(mode="fixed", keep_p=0.15))
    assert rc == 0
    # the quantised logits scratch of all 12 slabs (32 rows x 16 bits per
    # token) is the dominant term
    assert 12 * 32768 * 32 * 2 <= n < 12 * 32768 * 32 * 4


def test_kernels_per_call(lib):
    # one wave of 12 slabs: prep, logits, importance, pool sums, rank, gather
    assert sp.kernels_per_call(_shape(), sp.SelectionParams(mode="fixed", keep_p=0.15)) == 6
    # a pool window wider than the fused kernel's halo takes the staged path
    # (pool, chunk, select, gather scan instead of pool sums + post)
    assert sp.kernels_per_call(_shape(), sp.SelectionParams(pool_w=201)) == 8
    n = ctypes.c_int()
    assert lib.sp_kernels_per_call(ctypes.byref(_shape(head_dim=96)),
                                   ctypes.byref(sp.SelectionParams()._c()), ctypes.byref(n)) == 2


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), 2),          # unsupported head_dim
    (dict(n_q_heads=6, n_kv_heads=4), 1),  # Hq not a multiple of Hk
    (dict(n_lookahead=17), 2),       # L*G = 68 > 64 rows
    (dict(n_tokens_total=0), 1),
    (dict(n_seqs=0), 1),
])
def test_bad_shapes_rejected(lib, kw, code):
    rc, _ = _ws(_shape(**kw), sp.SelectionParams())
    assert rc == code


@pytest.mark.parametrize("kw", [
    dict(pool_w=12), dict(pool_w=0), dict(chunk=0), dict(mode="fixed", keep_p=0.0),
    dict(mode="fixed", keep_p=1.5), dict(mode="mass", mass=0.0), dict(boost_first_mult=0.0),
    dict(boost_last_n=-1), dict(scale=-1.0), dict(min_tok=-1), dict(max_keep=-1),
])
def test_bad_params_rejected(lib, kw):
    rc, _ = _ws(_shape(), sp.SelectionParams(**kw))
    assert rc == 1


def test_misaligned_stride_rejected(lib):
    s = _shape()
    s.k_stride_token = 2 * 256 + 4   # 1032 bytes: not a multiple of 16
    rc, _ = _ws(s, sp.SelectionParams())
    assert rc == 2


def test_null_pointers_rejected_before_any_launch(lib):
    s, p = _shape(), sp.SelectionParams()
    rc = lib.sp_attn_importance(ctypes.byref(s), ctypes.byref(p._c()), None, None, None, None,
                                None, 0, None)
    assert rc == 1
    rc = lib.sp_get_device_status(None, 0, None, 0, None)
    assert rc == 1


def test_workspace_checks(lib):
    s, p = _shape(n_tokens_total=512), sp.SelectionParams()
    buf = (ctypes.c_uint8 * 1024)()
    rc = lib.sp_workspace_init(None, 0, None)
    assert rc == 3
    rc = lib.sp_workspace_init(ctypes.addressof(buf) | 1, 512, None)
    assert rc == 3


def test_gather_rows_and_tokens_validate_on_the_host(lib):
    """Bad sizes, strides, alignment and null pointers are refused before any
    launch; the pointers below are never dereferenced."""
    a = ctypes.c_void_p(4096)
    s = _shape(n_tokens_total=1024)
    ok_rows = 1024

    def rows(shape, src=a, dst=a, dst_rows=ok_rows, idx=a, nk=a):
        return lib.sp_gather_rows(ctypes.byref(shape) if shape is not None else None, idx, nk,
                                  src, dst, dst_rows, None)

    assert rows(None) == 1
    assert rows(s, idx=None) == 1
    assert rows(s, nk=None) == 1
    assert rows(s, src=None) == 1
    assert rows(s, dst_rows=1023) == 1                      # fewer rows than tokens
    assert rows(s, src=ctypes.c_void_p(4096 + 8)) == 1      # src not 16-byte aligned
    assert rows(s, dst=ctypes.c_void_p(4096 + 2)) == 1
    bad = _shape(n_tokens_total=1024, head_dim=60)           # d not a whole number of vectors
    assert rows(bad) == 1
    bad = _shape(n_tokens_total=1024)
    bad.k_stride_token = 2 * 256 + 4                         # token stride not 16-byte multiple
    assert rows(bad) == 1
    bad = _shape(n_tokens_total=1024)
    bad.k_stride_head = 128                                   # heads overlap
    assert rows(bad) == 1
    bad = _shape(n_tokens_total=0)
    assert rows(bad, dst_rows=0) == 1
    assert lib.sp_gather_tokens(None, 16, a, a, a, None) == 1
    assert lib.sp_gather_tokens(a, 0, a, a, a, None) == 1
    assert lib.sp_gather_tokens(a, 16, a, a, None, None) == 1
    assert lib.sp_gather_tokens(a, (1 << 30) + 1, a, a, a, None) == 1


def test_listing_rule_validation(lib):
    s = _shape()
    bad = sp.SelectionParams()._c()
    bad.rule = 2
    n = ctypes.c_size_t()
    assert lib.sp_workspace_size(ctypes.byref(s), ctypes.byref(bad), ctypes.byref(n)) == 1
    a = ctypes.c_void_p(4096)
    listing = sp.SelectionParams(rule="listing", mode="fixed", keep_p=0.3)._c()
    # chunk-level stage entry points do not take the token-level listing rule
    assert lib.sp_select(ctypes.byref(s), ctypes.byref(listing), a, a, a, a, a, 1 << 30, None) == 2
    assert lib.sp_gather_kept(ctypes.byref(s), ctypes.byref(listing), a, a, a, a, a, a, a, a,
                              1 << 30, None) == 2
    # the listing rule runs on the fused post path only (chunk dividing 128)
    odd = sp.SelectionParams(rule="listing", chunk=48)._c()
    assert lib.sp_specprefill_score(ctypes.byref(s), ctypes.byref(odd), a, a, a, None, None, None,
                                    None, None, a, a, a, a, a, 1 << 30, None, None) == 2
    assert lib.sp_select_from_importance(ctypes.byref(s), ctypes.byref(odd), a, a, None, None, None,
                                         None, a, a, a, a, a, 1 << 30, None) == 2
    # same kernel count as the exact rule (its own gather kernel)
    assert sp.kernels_per_call(s, sp.SelectionParams(rule="listing", mode="fixed")) == 6


def test_auto_window_matches_the_oracle(lib):
    import oracle
    for spec_ctx in (130, 200, 600, 640, 1024, 2048, 4096, 8192, 16384, 32768, 131072):
        for req in (0, -5, 100, 512, 1000, 3000, 100000):
            assert sp.auto_window(spec_ctx, req) == oracle.auto_window(spec_ctx, req), (spec_ctx, req)
    w = ctypes.c_int32()
    assert lib.sp_auto_window(129, 0, ctypes.byref(w), ctypes.byref(w)) == 1
    assert lib.sp_auto_window(8192, 0, None, ctypes.byref(w)) == 1


def test_window_plan_matches_the_oracle(lib):
    import numpy as np
    import oracle
    rng = np.random.default_rng(4)
    cases = [(10000, 2000, 1000), (4500, 2000, 1000), (1500, 2000, 1000), (0, 2000, 1000),
             (2000, 2000, 1000), (2001, 2000, 1000), (7, 3, 1)]
    cases += [(int(rng.integers(0, 5000)), int(w), int(w) // 2) for w in rng.integers(2, 900, 40)]
    for n, window, stride in cases:
        assert sp.window_plan(n, window, stride) == oracle.window_plan(n, window, stride), (n, window)
    # a short buffer receives the first windows, the count is the full one
    cnt = ctypes.c_int32()
    arr = [(ctypes.c_int32 * 2)() for _ in range(3)]
    assert lib.sp_window_plan(10000, 2000, 1000, *[ctypes.addressof(x) for x in arr], 2,
                              ctypes.byref(cnt)) == 0
    assert cnt.value == 9 and list(arr[0]) == [0, 1000] and list(arr[2]) == [1000, 1000]
    for bad in ((100, 10, 0), (100, 10, 11), (-1, 10, 5)):
        assert lib.sp_window_plan(*bad, None, None, None, 0, ctypes.byref(cnt)) == 1
    assert lib.sp_window_plan(100, 10, 5, None, None, None, 4, ctypes.byref(cnt)) == 1
    assert lib.sp_merge_windows(100, 10, 0, ctypes.c_void_p(4096), ctypes.c_void_p(4096), None) == 1
    assert lib.sp_merge_windows(100, 10, 5, None, ctypes.c_void_p(4096), None) == 1


def test_pool_at_validation(lib):
    s = _shape()
    bad = sp.SelectionParams()._c()
    bad.pool_at = 2
    n = ctypes.c_size_t()
    assert lib.sp_workspace_size(ctypes.byref(s), ctypes.byref(bad), ctypes.byref(n)) == 1
    # per-head pooling keeps its halo in shared memory: half window <= 64
    rc, _ = _ws(s, sp.SelectionParams(pool_at="head", pool_w=131))
    assert rc == 2
    rc, _ = _ws(s, sp.SelectionParams(pool_at="head", pool_w=129))
    assert rc == 0
    # the pool is applied before the max, so the post path sees width 1: its
    # fused kernels only need the chunk to divide 128
    assert sp.kernels_per_call(s, sp.SelectionParams(pool_at="head", pool_w=129, chunk=48)) == 8
    assert sp.kernels_per_call(s, sp.SelectionParams(pool_at="head", pool_w=129)) == 6
    assert sp.kernels_per_call(s, sp.SelectionParams(pool_at="token", pool_w=131)) == 8


def test_kv_source_validation(lib):
    """Draft-cache key sources are checked on the host before any launch."""
    s = _shape(n_tokens_total=4096, n_layers=2)
    p = sp.SelectionParams()._c()
    a = ctypes.c_void_p(4096)

    def call(ptrs, table=None, bs=0, stride=0, rows=4096, shape=s):
        # a 16-byte workspace: every call that passes the checks stops there
        arr = (ctypes.c_void_p * len(ptrs))(*ptrs)
        src = sp._KvSource(ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), table, bs, stride, rows)
        return lib.sp_specprefill_score_kv(ctypes.byref(shape), ctypes.byref(p), a, a, ctypes.byref(src),
                                           None, None, None, None, None, a, a, a, a, a, 16, None)

    good = [8192, 12288]
    assert lib.sp_specprefill_score_kv(ctypes.byref(s), ctypes.byref(p), a, a, None, None, None,
                                       None, None, None, a, a, a, a, a, 1 << 40, None) == 1
    assert call([8192, None]) == 1                     # a missing layer pool
    assert call([8192, 12296]) == 1                    # not 16-byte aligned
    assert call(good, rows=4095) == 1                  # pool shorter than the packed tokens
    assert call(good, table=4096, bs=12, stride=8) == 1     # unsupported block size
    assert call(good, table=4096, bs=16, stride=0) == 1     # empty table rows
    assert call(good, table=4096, bs=16, stride=8, rows=1 << 31) == 1  # rows past int32
    many = _shape(n_tokens_total=4096, n_layers=65)
    assert call([8192] * 65, shape=many) == 2          # more layers than tensor maps
    # the workspace check comes after: a valid source reaches it
    assert call(good, table=4096, bs=16, stride=256) == 3


def test_noalloc_rejects_an_oversized_batch_before_any_launch(lib):
    """The fixed scratch of sp_pool_chunk_noalloc holds the offset tables and
    one (min, max) pair per pooling block; a batch that does not fit is
    refused on the host (the pointers are never dereferenced)."""
    a = ctypes.c_void_p(4096)
    p = sp.SelectionParams(mode="mass")._c()
    # 65536 prompts: four tables of 256 KB each do not fit 1 MiB
    big_b = sp.token_shape(65536, 1 << 20)
    assert lib.sp_pool_chunk_noalloc(ctypes.byref(big_b), ctypes.byref(p), a, a, a, a, a, None,
                                     None) == 2
    # 2^30 tokens at chunk 32: 2^20 pooling blocks of 8 bytes
    big_n = sp.token_shape(1, 1 << 30)
    assert lib.sp_pool_chunk_noalloc(ctypes.byref(big_n), ctypes.byref(p), a, a, a, a, a, None,
                                     None) == 2
    # null outputs are refused first
    ok = sp.token_shape(4, 4096)
    assert lib.sp_pool_chunk_noalloc(ctypes.byref(ok), ctypes.byref(p), a, a, None, a, a, None,
                                     None) == 1


def test_wave_budget_parameter(lib):
    """sp_params.wave_mib bounds one wave's logits scratch: the default keeps
    a 65K-token, 16-slab batch in one wave, 80 MiB splits it in two (one
    more logits and importance kernel), a negative budget is invalid."""
    s = _shape(n_seqs=1, n_layers=4, n_q_heads=16, n_kv_heads=4, head_dim=64, n_lookahead=16,
               n_tokens_total=65536)
    assert sp.kernels_per_call(s, sp.SelectionParams()) == 6
    assert sp.kernels_per_call(s, sp.SelectionParams(wave_mib=80)) == 8
    rc, small = _ws(s, sp.SelectionParams(wave_mib=80))
    rc0, big = _ws(s, sp.SelectionParams())
    assert rc == rc0 == 0 and small < big
    rc, _ = _ws(s, sp.SelectionParams(wave_mib=-1))
    assert rc == 1
