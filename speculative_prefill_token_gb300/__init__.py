"""Python binding of libspecprefill (the SpecPrefill scoring path on sm_103a).

Argument marshalling only: every step of the path runs in the CUDA library
through its C ABI (include/specprefill.h). PyTorch supplies device memory and
streams. There is no CPU fallback: if the library is missing or fails to
load, every call raises.

Tensor conventions (bf16 data carried as torch.bfloat16 or as uint16 bits):
  q        [B, Ly, L, Hq, d]   lookahead queries of each prompt (strided ok,
                               head_dim contiguous)
  k        [Ly, Ntot, Hk, d]   token-major key cache of the packed prompts
  seq_off  [B+1] int32         prompt offsets on the token axis
"""

import ctypes
import os
from dataclasses import dataclass, field
from typing import Optional

__all__ = [
    "SelectionParams",
    "SpecPrefillError",
    "load",
    "lib",
    "workspace_size",
    "max_chunks",
    "make_workspace",
    "attn_importance",
    "attn_importance_simt",
    "pool_chunk",
    "pool_chunk_noalloc",
    "select",
    "gather_kept",
    "gather_rows",
    "gather_tokens",
    "select_from_importance",
    "kv_source",
    "specprefill_score_kv",
    "attn_importance_kv",
    "auto_window",
    "window_plan",
    "merge_windows",
    "specprefill_score",
    "device_status",
    "STATUS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecprefill.so")

STATUS = {0: "SP_OK", 1: "SP_ERR_INVALID_ARG", 2: "SP_ERR_UNSUPPORTED", 3: "SP_ERR_WORKSPACE",
          4: "SP_ERR_CUDA", 5: "SP_ERR_TIMEOUT", 6: "SP_ERR_DEVICE"}
MODES = {"fixed": 0, "mass": 1}
RULES = {"exact": 0, "listing": 1}
POOL_AT = {"token": 0, "head": 1}


class SpecPrefillError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


class _Shape(ctypes.Structure):
    _fields_ = [("n_seqs", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_lookahead", ctypes.c_int32),
                ("n_tokens_total", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("k_stride_layer", ctypes.c_int64), ("k_stride_token", ctypes.c_int64),
                ("k_stride_head", ctypes.c_int64), ("q_stride_seq", ctypes.c_int64),
                ("q_stride_layer", ctypes.c_int64), ("q_stride_step", ctypes.c_int64),
                ("q_stride_head", ctypes.c_int64)]


class _Params(ctypes.Structure):
    _fields_ = [("pool_w", ctypes.c_int32), ("chunk", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("keep_p", ctypes.c_float), ("mass", ctypes.c_float),
                ("normalize", ctypes.c_int32), ("boost_first_mult", ctypes.c_float),
                ("boost_first_n", ctypes.c_int32), ("boost_last_mult", ctypes.c_float),
                ("boost_last_n", ctypes.c_int32), ("force_bos", ctypes.c_int32),
                ("force_last_chunk", ctypes.c_int32), ("scale", ctypes.c_float),
                ("spin_limit", ctypes.c_int32), ("rule", ctypes.c_int32),
                ("min_tok", ctypes.c_int32), ("max_keep", ctypes.c_int32),
                ("pool_at", ctypes.c_int32), ("wave_mib", ctypes.c_int32)]


class _KvSource(ctypes.Structure):
    _fields_ = [("layer_k", ctypes.POINTER(ctypes.c_void_p)), ("block_table", ctypes.c_void_p),
                ("block_size", ctypes.c_int32), ("table_stride", ctypes.c_int32),
                ("pool_tokens", ctypes.c_int64)]


class _Profile(ctypes.Structure):
    _fields_ = [("logits_start", ctypes.c_void_p), ("logits_stop", ctypes.c_void_p)]


@dataclass
class SelectionParams:
    """Selection settings; defaults are the pages' (W=13, C=32, mass 0.85,
    boost x1.5 first 64 / x1.3 last 128, BOS and final chunk kept).
    rule "listing" selects like the pages' own tool (ties at the threshold,
    tokens {0,1,2,3,n-2,n-1}, fill to min(min_tok, max(4, n/10)), cap to
    max_keep tokens when max_keep > 0). pool_at "head" pools every attention
    row before the max over heads and layers instead of the per-token
    importance. wave_mib (0: the library's default) bounds the logits
    scratch of one wave in MiB; larger batches are scored in several
    waves."""
    pool_w: int = 13
    chunk: int = 32
    mode: str = "mass"
    keep_p: float = 0.30
    mass: float = 0.85
    normalize: bool = True
    boost_first_mult: float = 1.5
    boost_first_n: int = 64
    boost_last_mult: float = 1.3
    boost_last_n: int = 128
    force_bos: bool = True
    force_last_chunk: bool = True
    scale: float = 0.0
    spin_limit: int = 0
    rule: str = "exact"
    min_tok: int = 128
    max_keep: int = 0
    pool_at: str = "token"
    wave_mib: int = 0

    def _c(self) -> _Params:
        return _Params(int(self.pool_w), int(self.chunk), MODES[self.mode], float(self.keep_p),
                       float(self.mass), int(bool(self.normalize)), float(self.boost_first_mult),
                       int(self.boost_first_n), float(self.boost_last_mult), int(self.boost_last_n),
                       int(bool(self.force_bos)), int(bool(self.force_last_chunk)),
                       float(self.scale), int(self.spin_limit), RULES[self.rule],
                       int(self.min_tok), int(self.max_keep), POOL_AT[self.pool_at], int(self.wave_mib))


_lib = None
_P = ctypes.c_void_p
_SZ = ctypes.c_size_t


def load(path: Optional[str] = None):
    """Load the shared library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"libspecprefill.so not built ({path}); run __graft_entry__.build()")
    lib_ = ctypes.CDLL(path)
    sp = ctypes.POINTER(_Shape)
    pp = ctypes.POINTER(_Params)
    i32 = ctypes.c_int
    sigs = {
        "sp_max_chunks": [sp, pp, ctypes.POINTER(ctypes.c_int64)],
        "sp_kernels_per_call": [sp, pp, ctypes.POINTER(i32)],
        "sp_workspace_size": [sp, pp, ctypes.POINTER(_SZ)],
        "sp_workspace_init": [_P, _SZ, _P],
        "sp_attn_importance": [sp, pp, _P, _P, _P, _P, _P, _SZ, _P],
        "sp_attn_importance_simt": [sp, pp, _P, _P, _P, _P, _P, _SZ, _P],
        "sp_pool_chunk": [sp, pp, _P, _P, _P, _P, _P, _P, _SZ, _P],
        "sp_pool_chunk_noalloc": [sp, pp, _P, _P, _P, _P, _P, _P, _P],
        "sp_select": [sp, pp, _P, _P, _P, _P, _P, _SZ, _P],
        "sp_gather_kept": [sp, pp, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
        "sp_specprefill_score": [sp, pp, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                 _P, ctypes.POINTER(_Profile)],
        "sp_gather_rows": [sp, _P, _P, _P, _P, ctypes.c_int64, _P],
        "sp_select_from_importance": [sp, pp, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
        "sp_auto_window": [i32, i32, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)],
        "sp_window_plan": [ctypes.c_int64, i32, i32, _P, _P, _P, i32, ctypes.POINTER(ctypes.c_int32)],
        "sp_merge_windows": [ctypes.c_int64, i32, i32, _P, _P, _P],
        "sp_gather_tokens": [_P, ctypes.c_int64, _P, _P, _P, _P],
        "sp_attn_importance_kv": [sp, pp, _P, _P, ctypes.POINTER(_KvSource), _P, _P, _SZ, _P],
        "sp_specprefill_score_kv": [sp, pp, _P, _P, ctypes.POINTER(_KvSource), _P, _P, _P, _P, _P, _P,
                                    _P, _P, _P, _P, _SZ, _P],
        "sp_get_device_status": [_P, _SZ, _P, i32, ctypes.POINTER(ctypes.c_int32)],
    }
    for name, args in sigs.items():
        fn = getattr(lib_, name)
        fn.argtypes = args
        fn.restype = i32
    lib_.sp_status_string.argtypes = [i32]
    lib_.sp_status_string.restype = ctypes.c_char_p
    lib_.sp_build_info.argtypes = []
    lib_.sp_build_info.restype = ctypes.c_char_p
    _lib = lib_
    return _lib


def lib():
    return load()


def _check(rc: int, what: str):
    if rc != 0:
        raise SpecPrefillError(rc, what)


# ---------------------------------------------------------------- marshalling


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def shape_of(q, k, seq_off=None, n_seqs: Optional[int] = None, max_seq_len: int = 0) -> _Shape:
    """C shape struct from the q [B, Ly, L, Hq, d] and k [Ly, Ntot, Hk, d]
    tensors; max_seq_len > 0 states the longest prompt allowed (a longer one
    makes the call's device status SP_ERR_DEVICE)."""
    if q.dim() != 5 or k.dim() != 4:
        raise ValueError("q must be [B, Ly, L, Hq, d] and k [Ly, Ntot, Hk, d]")
    if q.element_size() != 2 or k.element_size() != 2:
        raise ValueError("q and k must hold bf16 (torch.bfloat16 or uint16 bits)")
    b, ly, steps, hq, d = q.shape
    ly_k, ntot, hk, d_k = k.shape
    if ly_k != ly or d_k != d:
        raise ValueError("q and k disagree on layers or head_dim")
    if q.stride(-1) != 1 or k.stride(-1) != 1:
        raise ValueError("head_dim must be contiguous")
    return _Shape(int(b), int(ly), int(hq), int(hk), int(d), int(steps), int(ntot), int(max_seq_len),
                  k.stride(0), k.stride(1), k.stride(2),
                  q.stride(0), q.stride(1), q.stride(2), q.stride(3))


def token_shape(n_seqs: int, n_tokens_total: int, n_layers=1, n_q_heads=1, n_kv_heads=1,
                head_dim=64, n_lookahead=1) -> _Shape:
    """Shape struct for the stages that only need the token axis (pool,
    select, gather); the attention dimensions are placeholders."""
    return _Shape(int(n_seqs), n_layers, n_q_heads, n_kv_heads, head_dim, n_lookahead,
                  int(n_tokens_total), 0, head_dim * n_tokens_total * n_kv_heads,
                  head_dim * n_kv_heads, head_dim, head_dim, head_dim, head_dim, head_dim)


def workspace_size(shape: _Shape, params: SelectionParams) -> int:
    n = _SZ()
    _check(lib().sp_workspace_size(ctypes.byref(shape), ctypes.byref(params._c()), ctypes.byref(n)),
           "sp_workspace_size")
    return int(n.value)


def max_chunks(shape: _Shape, params: SelectionParams) -> int:
    n = ctypes.c_int64()
    _check(lib().sp_max_chunks(ctypes.byref(shape), ctypes.byref(params._c()), ctypes.byref(n)),
           "sp_max_chunks")
    return int(n.value)


def kernels_per_call(shape: _Shape, params: SelectionParams) -> int:
    """Kernels one specprefill_score call launches (all of them this library's)."""
    n = ctypes.c_int()
    _check(lib().sp_kernels_per_call(ctypes.byref(shape), ctypes.byref(params._c()),
                                     ctypes.byref(n)), "sp_kernels_per_call")
    return int(n.value)


def make_workspace(shape: _Shape, params: SelectionParams, device=None, poison: bool = False):
    """Allocate (torch) and initialise a workspace for this shape. With
    ``poison`` every byte except the header starts as 0xFF (NaN as float)."""
    import torch
    nbytes = workspace_size(shape, params)
    ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + nbytes]
    if poison:
        ws.fill_(0xFF)
    _check(lib().sp_workspace_init(ws.data_ptr(), nbytes, _stream(None)), "sp_workspace_init")
    return ws


def _ws_args(ws):
    return ws.data_ptr(), ws.numel()


def attn_importance(q, k, seq_off, params: SelectionParams, imp=None, ws=None, stream=None,
                    simt: bool = False):
    """imp[t] for every packed token (float32, device)."""
    import torch
    shape = shape_of(q, k)
    if imp is None:
        imp = torch.empty(shape.n_tokens_total, dtype=torch.float32, device=k.device)
    if ws is None:
        ws = make_workspace(shape, params, k.device)
    fn = lib().sp_attn_importance_simt if simt else lib().sp_attn_importance
    _check(fn(ctypes.byref(shape), ctypes.byref(params._c()), seq_off.data_ptr(), q.data_ptr(),
              k.data_ptr(), imp.data_ptr(), *_ws_args(ws), _stream(stream)),
           "sp_attn_importance")
    return imp


def attn_importance_simt(q, k, seq_off, params: SelectionParams, imp=None, ws=None, stream=None):
    return attn_importance(q, k, seq_off, params, imp, ws, stream, simt=True)


def pool_chunk(imp, seq_off, params: SelectionParams, tok_score=None, ws=None, stream=None):
    """(tok_score, chunk_score, chunk_off) from imp."""
    import torch
    n_seqs = seq_off.numel() - 1
    shape = token_shape(n_seqs, imp.numel())
    nch = max_chunks(shape, params)
    chunk_score = torch.empty(nch, dtype=torch.float32, device=imp.device)
    chunk_off = torch.empty(n_seqs + 1, dtype=torch.int32, device=imp.device)
    if ws is None:
        ws = make_workspace(shape, params, imp.device)
    _check(lib().sp_pool_chunk(ctypes.byref(shape), ctypes.byref(params._c()), seq_off.data_ptr(),
                               imp.data_ptr(), _ptr(tok_score), chunk_score.data_ptr(),
                               chunk_off.data_ptr(), *_ws_args(ws), _stream(stream)),
           "sp_pool_chunk")
    return tok_score, chunk_score, chunk_off


def pool_chunk_noalloc(imp, seq_off, params: SelectionParams, tok_score, chunk_score, chunk_off,
                       status=None, stream=None):
    """sp_pool_chunk without a workspace (fixed scratch inside the library);
    all outputs are caller-provided. For callers that cannot allocate device
    memory at call time."""
    shape = token_shape(seq_off.numel() - 1, imp.numel())
    _check(lib().sp_pool_chunk_noalloc(ctypes.byref(shape), ctypes.byref(params._c()),
                                       seq_off.data_ptr(), imp.data_ptr(), tok_score.data_ptr(),
                                       chunk_score.data_ptr(), chunk_off.data_ptr(), _ptr(status),
                                       _stream(stream)), "sp_pool_chunk_noalloc")


def select(chunk_score, chunk_off, seq_off, n_tokens_total: int, params: SelectionParams,
           ws=None, stream=None):
    """uint8 chunk_keep (bit 0 ranked, bit 1 forced final chunk)."""
    import torch
    n_seqs = seq_off.numel() - 1
    shape = token_shape(n_seqs, n_tokens_total)
    keep = torch.zeros(chunk_score.numel(), dtype=torch.uint8, device=chunk_score.device)
    if ws is None:
        ws = make_workspace(shape, params, chunk_score.device)
    _check(lib().sp_select(ctypes.byref(shape), ctypes.byref(params._c()), seq_off.data_ptr(),
                           chunk_off.data_ptr(), chunk_score.data_ptr(), keep.data_ptr(),
                           *_ws_args(ws), _stream(stream)), "sp_select")
    return keep


def gather_kept(chunk_keep, chunk_off, seq_off, n_tokens_total: int, params: SelectionParams,
                ws=None, stream=None):
    """(kept_idx, kept_pos, kept_off, n_kept) device tensors; the lists hold
    n_kept valid entries (capacity n_tokens_total)."""
    import torch
    n_seqs = seq_off.numel() - 1
    shape = token_shape(n_seqs, n_tokens_total)
    dev = chunk_keep.device
    kept_idx = torch.empty(n_tokens_total, dtype=torch.int32, device=dev)
    kept_pos = torch.empty(n_tokens_total, dtype=torch.int32, device=dev)
    kept_off = torch.empty(n_seqs + 1, dtype=torch.int32, device=dev)
    n_kept = torch.empty(1, dtype=torch.int32, device=dev)
    if ws is None:
        ws = make_workspace(shape, params, dev)
    _check(lib().sp_gather_kept(ctypes.byref(shape), ctypes.byref(params._c()), seq_off.data_ptr(),
                                chunk_off.data_ptr(), chunk_keep.data_ptr(), kept_idx.data_ptr(),
                                kept_pos.data_ptr(), kept_off.data_ptr(), n_kept.data_ptr(),
                                *_ws_args(ws), _stream(stream)), "sp_gather_kept")
    return kept_idx, kept_pos, kept_off, n_kept


def gather_rows(cache, kept_idx, n_kept, out=None, stream=None):
    """Rows of the kept tokens of a token-major bf16 cache tensor
    ``[Ly][Ntot][Hk][d]`` (any strides, d contiguous), packed into ``out``
    (dense ``[Ly][R][Hk][d]``, R >= Ntot, allocated with R = Ntot when
    omitted): out[l, i] = cache[l, kept_idx[i]] for i < n_kept. Rows past
    n_kept are left untouched."""
    import torch
    if cache.dtype != torch.bfloat16 or cache.dim() != 4 or cache.stride(-1) != 1:
        raise ValueError("cache must be a bf16 [Ly][Ntot][Hk][d] tensor with d contiguous")
    ly, ntot, hk, d = cache.shape
    if out is None:
        out = torch.empty(ly, ntot, hk, d, dtype=cache.dtype, device=cache.device)
    if (out.dtype != cache.dtype or out.dim() != 4 or not out.is_contiguous()
            or out.shape[0] != ly or out.shape[2:] != cache.shape[2:]):
        raise ValueError("out must be a dense bf16 [Ly][R][Hk][d] tensor")
    shape = _Shape(1, int(ly), int(hk), int(hk), int(d), 1, int(ntot), 0,
                   cache.stride(0), cache.stride(1), cache.stride(2), d, d, d, d)
    _check(lib().sp_gather_rows(ctypes.byref(shape), kept_idx.data_ptr(), n_kept.data_ptr(),
                                cache.data_ptr(), out.data_ptr(), int(out.shape[1]),
                                _stream(stream)), "sp_gather_rows")
    return out


def gather_tokens(token_ids, kept_idx, n_kept, out=None, stream=None):
    """Kept token ids for the target's batch: out[i] = token_ids[kept_idx[i]]
    for i < n_kept (int32, device)."""
    import torch
    n = token_ids.numel()
    if token_ids.dtype != torch.int32 or not token_ids.is_contiguous():
        raise ValueError("token_ids must be a contiguous int32 tensor")
    if out is None:
        out = torch.empty(n, dtype=torch.int32, device=token_ids.device)
    if out.dtype != torch.int32 or out.numel() < n or not out.is_contiguous():
        raise ValueError("out must be a contiguous int32 tensor of at least len(token_ids)")
    _check(lib().sp_gather_tokens(token_ids.data_ptr(), int(n), kept_idx.data_ptr(),
                                  n_kept.data_ptr(), out.data_ptr(), _stream(stream)),
           "sp_gather_tokens")
    return out


@dataclass
class ScoreOutputs:
    kept_idx: object
    kept_pos: object
    kept_off: object
    n_kept: object
    imp: object = None
    tok_score: object = None
    chunk_score: object = None
    chunk_off: object = None
    chunk_keep: object = None


def alloc_outputs(q, k, params: SelectionParams, intermediates: bool = True) -> ScoreOutputs:
    import torch
    shape = shape_of(q, k)
    dev = k.device
    ntot, nb = shape.n_tokens_total, shape.n_seqs
    out = ScoreOutputs(kept_idx=torch.empty(ntot, dtype=torch.int32, device=dev),
                       kept_pos=torch.empty(ntot, dtype=torch.int32, device=dev),
                       kept_off=torch.empty(nb + 1, dtype=torch.int32, device=dev),
                       n_kept=torch.empty(1, dtype=torch.int32, device=dev))
    if intermediates:
        nch = max_chunks(shape, params)
        out.imp = torch.empty(ntot, dtype=torch.float32, device=dev)
        out.tok_score = torch.empty(ntot, dtype=torch.float32, device=dev)
        out.chunk_score = torch.empty(nch, dtype=torch.float32, device=dev)
        out.chunk_off = torch.empty(nb + 1, dtype=torch.int32, device=dev)
        out.chunk_keep = torch.empty(nch, dtype=torch.uint8, device=dev)
    return out


def specprefill_score(q, k, seq_off, params: SelectionParams, out: Optional[ScoreOutputs] = None,
                      ws=None, stream=None, profile_events=None, max_seq_len: int = 0) -> ScoreOutputs:
    """The whole path: kept token indices and positions per prompt.

    ``profile_events`` = (start, stop) torch.cuda.Event pair recorded around
    the logits kernel(s). ``max_seq_len`` > 0: the longest prompt allowed.
    """
    shape = shape_of(q, k, max_seq_len=max_seq_len)
    if out is None:
        out = alloc_outputs(q, k, params)
    if ws is None:
        ws = make_workspace(shape, params, k.device)
    prof = None
    if profile_events is not None:
        prof = ctypes.byref(_Profile(profile_events[0].cuda_event, profile_events[1].cuda_event))
    _check(lib().sp_specprefill_score(
        ctypes.byref(shape), ctypes.byref(params._c()), seq_off.data_ptr(), q.data_ptr(),
        k.data_ptr(), _ptr(out.imp), _ptr(out.tok_score), _ptr(out.chunk_score),
        _ptr(out.chunk_off), _ptr(out.chunk_keep), out.kept_idx.data_ptr(),
        out.kept_pos.data_ptr(), out.kept_off.data_ptr(), out.n_kept.data_ptr(), *_ws_args(ws),
        _stream(stream), prof), "sp_specprefill_score")
    return out


def select_from_importance(imp, seq_off, params: SelectionParams, out: Optional[ScoreOutputs] = None,
                           ws=None, stream=None) -> ScoreOutputs:
    """Pooling, normalisation, boost, chunk scores, selection and kept lists
    from a given per-token importance (float32, device). ``out.imp`` is the
    given ``imp``."""
    import torch
    n_seqs = seq_off.numel() - 1
    ntot = imp.numel()
    shape = token_shape(n_seqs, ntot)
    dev = imp.device
    if out is None:
        nch = max_chunks(shape, params)
        out = ScoreOutputs(kept_idx=torch.empty(ntot, dtype=torch.int32, device=dev),
                           kept_pos=torch.empty(ntot, dtype=torch.int32, device=dev),
                           kept_off=torch.empty(n_seqs + 1, dtype=torch.int32, device=dev),
                           n_kept=torch.empty(1, dtype=torch.int32, device=dev),
                           tok_score=torch.empty(ntot, dtype=torch.float32, device=dev),
                           chunk_score=torch.empty(nch, dtype=torch.float32, device=dev),
                           chunk_off=torch.empty(n_seqs + 1, dtype=torch.int32, device=dev),
                           chunk_keep=torch.empty(nch, dtype=torch.uint8, device=dev))
    out.imp = imp
    if ws is None:
        ws = make_workspace(shape, params, dev)
    _check(lib().sp_select_from_importance(
        ctypes.byref(shape), ctypes.byref(params._c()), seq_off.data_ptr(), imp.data_ptr(),
        _ptr(out.tok_score), _ptr(out.chunk_score), _ptr(out.chunk_off), _ptr(out.chunk_keep),
        out.kept_idx.data_ptr(), out.kept_pos.data_ptr(), out.kept_off.data_ptr(),
        out.n_kept.data_ptr(), *_ws_args(ws), _stream(stream)), "sp_select_from_importance")
    return out


def auto_window(spec_ctx: int, window: int = 0):
    """(window, stride) of the sliding-window scoring for a draft context of
    spec_ctx tokens (host computation)."""
    w, st = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().sp_auto_window(int(spec_ctx), int(window), ctypes.byref(w), ctypes.byref(st)),
           "sp_auto_window")
    return int(w.value), int(st.value)


def window_plan(n: int, window: int, stride: int):
    """[(start, end, kept)] of the sliding-window scoring of an n-token prompt
    (host computation)."""
    cnt = ctypes.c_int32()
    _check(lib().sp_window_plan(int(n), int(window), int(stride), None, None, None, 0,
                                ctypes.byref(cnt)), "sp_window_plan")
    m = int(cnt.value)
    arr = [(ctypes.c_int32 * max(m, 1))() for _ in range(3)]
    _check(lib().sp_window_plan(int(n), int(window), int(stride), *[ctypes.addressof(a) for a in arr],
                                m, ctypes.byref(cnt)), "sp_window_plan")
    return [(arr[0][i], arr[1][i], arr[2][i]) for i in range(m)]


def merge_windows(imp_windows, n: int, window: int, stride: int, out=None, stream=None):
    """Per-token importance of an n-token prompt from its windows' importance
    vectors packed back to back (float32, device)."""
    import torch
    if imp_windows.dtype != torch.float32 or not imp_windows.is_contiguous():
        raise ValueError("imp_windows must be a contiguous float32 tensor")
    plan = window_plan(n, window, stride)
    need = sum(e - s for s, e, _ in plan)
    if imp_windows.numel() < need:
        raise ValueError(f"imp_windows holds {imp_windows.numel()} scores, the windows need {need}")
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=imp_windows.device)
    _check(lib().sp_merge_windows(int(n), int(window), int(stride), imp_windows.data_ptr(),
                                  out.data_ptr(), _stream(stream)), "sp_merge_windows")
    return out


def kv_source(layer_k, block_table=None, block_size: int = 0):
    """Key source over a draft engine's cache: ``layer_k`` is a list of one
    bf16 key pool per layer, each [rows, Hk, d] or, block-paged,
    [num_blocks, block_size, Hk, d] (d contiguous, rows evenly strided);
    ``block_table`` (int32, device, [B, max_blocks]) maps each prompt's
    logical blocks to pool blocks. Returns (struct, keep-alive, token stride,
    head stride, Hk, d)."""
    import torch
    k0 = layer_k[0]
    if k0.dim() == 4:
        nb, bs, hk, d = k0.shape
        if k0.stride(0) != bs * k0.stride(1):
            raise ValueError("blocks of a pool must follow one another with the token stride")
        rows, st_tok, st_head = nb * bs, k0.stride(1), k0.stride(2)
        if block_table is not None and block_size not in (0, bs):
            raise ValueError("block_size differs from the pools' block dimension")
        block_size = bs if block_table is not None else 0
    elif k0.dim() == 3:
        rows, hk, d = k0.shape
        st_tok, st_head = k0.stride(0), k0.stride(1)
    else:
        raise ValueError("each layer pool is [rows, Hk, d] or [blocks, block_size, Hk, d]")
    for kl in layer_k:
        if (kl.dtype != torch.bfloat16 or kl.shape != k0.shape or kl.stride() != k0.stride()
                or kl.stride(-1) != 1):
            raise ValueError("every layer pool must be bf16 with the first one's shape and strides")
    ptrs = (ctypes.c_void_p * len(layer_k))(*[kl.data_ptr() for kl in layer_k])
    table_stride = 0
    if block_table is not None:
        if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.stride(1) != 1:
            raise ValueError("block_table must be an int32 [B, max_blocks] tensor, rows contiguous")
        table_stride = block_table.stride(0)
    src = _KvSource(ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p)), _ptr(block_table),
                    int(block_size), int(table_stride), int(rows))
    return src, ptrs, int(st_tok), int(st_head), int(hk), int(d)


def shape_of_kv(q, layer_k, n_tokens_total: int, block_table=None) -> "_Shape":
    """Shape struct of a draft-cache call: Q as in shape_of, keys from the
    per-layer pools (their token and head strides)."""
    _, _, st_tok, st_head, hk, d = kv_source(layer_k, block_table)
    b, ly, steps, hq, dq = q.shape
    if dq != d or ly != len(layer_k):
        raise ValueError("q and the pools disagree on layers or head_dim")
    return _Shape(int(b), int(ly), int(hq), int(hk), int(d), int(steps), int(n_tokens_total), 0,
                  st_tok, st_tok, st_head, q.stride(0), q.stride(1), q.stride(2), q.stride(3))


def specprefill_score_kv(q, layer_k, seq_off, n_tokens_total: int, params: SelectionParams,
                         block_table=None, out: Optional[ScoreOutputs] = None, ws=None,
                         stream=None) -> ScoreOutputs:
    """The whole path with the keys read in place from per-layer (optionally
    block-paged) pools; n_tokens_total = seq_off[-1]."""
    import torch
    src, keep, *_ = kv_source(layer_k, block_table)
    shape = shape_of_kv(q, layer_k, n_tokens_total, block_table)
    dev = q.device
    if out is None:
        nb = shape.n_seqs
        nch = max_chunks(shape, params)
        out = ScoreOutputs(kept_idx=torch.empty(n_tokens_total, dtype=torch.int32, device=dev),
                           kept_pos=torch.empty(n_tokens_total, dtype=torch.int32, device=dev),
                           kept_off=torch.empty(nb + 1, dtype=torch.int32, device=dev),
                           n_kept=torch.empty(1, dtype=torch.int32, device=dev),
                           imp=torch.empty(n_tokens_total, dtype=torch.float32, device=dev),
                           tok_score=torch.empty(n_tokens_total, dtype=torch.float32, device=dev),
                           chunk_score=torch.empty(nch, dtype=torch.float32, device=dev),
                           chunk_off=torch.empty(nb + 1, dtype=torch.int32, device=dev),
                           chunk_keep=torch.empty(nch, dtype=torch.uint8, device=dev))
    if ws is None:
        ws = make_workspace(shape, params, dev)
    _check(lib().sp_specprefill_score_kv(
        ctypes.byref(shape), ctypes.byref(params._c()), seq_off.data_ptr(), q.data_ptr(),
        ctypes.byref(src), _ptr(out.imp), _ptr(out.tok_score), _ptr(out.chunk_score),
        _ptr(out.chunk_off), _ptr(out.chunk_keep), out.kept_idx.data_ptr(), out.kept_pos.data_ptr(),
        out.kept_off.data_ptr(), out.n_kept.data_ptr(), *_ws_args(ws), _stream(stream)),
        "sp_specprefill_score_kv")
    del keep
    return out


def attn_importance_kv(q, layer_k, seq_off, n_tokens_total: int, params: SelectionParams,
                       block_table=None, imp=None, ws=None, stream=None):
    """imp[t] for every packed token, keys read in place from the pools."""
    import torch
    src, keep, *_ = kv_source(layer_k, block_table)
    shape = shape_of_kv(q, layer_k, n_tokens_total, block_table)
    if imp is None:
        imp = torch.empty(n_tokens_total, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = make_workspace(shape, params, q.device)
    _check(lib().sp_attn_importance_kv(ctypes.byref(shape), ctypes.byref(params._c()),
                                       seq_off.data_ptr(), q.data_ptr(), ctypes.byref(src),
                                       imp.data_ptr(), *_ws_args(ws), _stream(stream)),
           "sp_attn_importance_kv")
    del keep
    return imp


def device_status(ws, stream=None, clear: bool = True) -> int:
    """Synchronise and read (and by default clear) the workspace status word."""
    v = ctypes.c_int32()
    _check(lib().sp_get_device_status(ws.data_ptr(), ws.numel(), _stream(stream), int(clear),
                                      ctypes.byref(v)), "sp_get_device_status")
    return int(v.value)
