"""Thin ctypes binding over libsv.so (the C ABI in include/sv.h).

Argument marshalling only: every step of the verify round runs in the
library's CUDA kernels.  Tensors must be CUDA tensors of the stated dtype,
contiguous; workspaces are allocated with torch when the caller passes none.
There is no fallback: if the library is missing or fails to load, importing
this module raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_F32 = ctypes.c_float
_SZ = ctypes.c_size_t


class SVError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


class _AttnShape(ctypes.Structure):
    _fields_ = [("B", _I32), ("R", _I32), ("Hq", _I32), ("Hkv", _I32), ("D", _I32), ("T_cap", _I32)]


def _load():
    if not os.path.exists(LIB):
        raise ImportError(f"libsv.so not built ({LIB}); run __graft_entry__.build() first")
    L = ctypes.CDLL(LIB)
    L.sv_version.restype = ctypes.c_int
    L.sv_status_string.restype = ctypes.c_char_p
    L.sv_status_string.argtypes = [ctypes.c_int]
    L.sv_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), _P]
    L.sv_verify_attn_workspace.argtypes = [ctypes.POINTER(_AttnShape)]
    L.sv_verify_attn_workspace.restype = _SZ
    L.sv_verify_attn.argtypes = [ctypes.POINTER(_AttnShape), _P, _P, _P, _P, _P, _P, _P, _F32, _P, _P, _SZ, _P]
    L.sv_lm_head_ex.argtypes = [_P, _P, _P, _I32, _I32, _I32, ctypes.c_uint32, _P]
    L.sv_verify_attn_ex.argtypes = [ctypes.POINTER(_AttnShape), _P, _P, _P, _P, _P, _P, _P, _F32, _P, _P, _SZ,
                                    ctypes.c_uint32, _P]
    L.sv_lm_head.argtypes = [_P, _P, _P, _I32, _I32, _I32, _P]
    L.sv_accept_greedy_workspace.argtypes = [_I32, _I32, _I32]
    L.sv_accept_greedy_workspace.restype = _SZ
    L.sv_accept_greedy.argtypes = [_P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _SZ, _P]
    L.sv_accept_greedy_relaxed_workspace.argtypes = [_I32, _I32, _I32]
    L.sv_accept_greedy_relaxed_workspace.restype = _SZ
    L.sv_accept_greedy_relaxed.argtypes = [_P, _P, _P, _I32, _I32, _I32, ctypes.c_float, _P, _P, _P, _P, _SZ, _P]
    L.sv_accept_sample_workspace.argtypes = [_I32, _I32, _I32]
    L.sv_accept_sample_workspace.restype = _SZ
    L.sv_accept_sample.argtypes = [_P, _P, _I32, _P, _P, _I32, _I32, _I32, _F32, _U64, _U64, _P, _P, _P, _P, _P,
                                   _SZ, _P]
    L.sv_accept_sample_noalloc.argtypes = [_P, _P, _I32, _P, _P, _I32, _I32, _I32, _F32, _U64, _U64, _P, _P, _P,
                                           _P, _P]
    L.sv_kv_commit.argtypes = [_P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P]
    L.sv_kv_commit_paged.argtypes = [_P, _P, _I32, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P]
    L.sv_verify_attn_paged.argtypes = [_P, _P, _P, _P, _I32, _P, _I32, _P, _P, _P, _P, ctypes.c_float, _P, _P, _SZ,
                                       ctypes.c_uint32, _P]
    L.sv_lm_head_argmax_bytes.argtypes = [_I32, _I32]
    L.sv_lm_head_argmax_bytes.restype = _SZ
    L.sv_lm_head_argmax.argtypes = [_P, _P, _P, _I32, _I32, _I32, _P, _SZ, ctypes.c_uint32, _P]
    L.sv_accept_greedy_commit.argtypes = [_P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32,
                                          _I32, _P, _P]
    L.sv_accept_greedy_commit_paged.argtypes = [_P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _I32, _P, _I32,
                                                _P, _P, _I32, _I32, _I32, _P, _P]
    L.sv_copy.argtypes = [_P, _P, _SZ, _P]
    L.sv_diag_exp.argtypes = [_P, _P, _I64, _P]
    L.sv_diag_div.argtypes = [_P, _P, _P, _I64, _P]
    L.sv_diag_philox.argtypes = [_P, _P, _P, _I64, _P]
    L.sv_diag_canon.argtypes = [_P, _I32, _I32, _P, _P, _P, _P]
    for fn in ("sv_verify_attn", "sv_verify_attn_ex", "sv_lm_head", "sv_lm_head_ex", "sv_accept_greedy",
               "sv_accept_greedy_relaxed", "sv_accept_sample",
               "sv_accept_sample_noalloc", "sv_kv_commit", "sv_kv_commit_paged", "sv_verify_attn_paged",
               "sv_diag_exp", "sv_diag_div", "sv_diag_philox", "sv_diag_canon", "sv_get_device_error", "sv_lm_head_argmax",
               "sv_accept_greedy_commit", "sv_accept_greedy_commit_paged", "sv_copy"):
        getattr(L, fn).restype = ctypes.c_int
    return L


lib = _load()


def _check(fn: str, status: int):
    if status != 0:
        raise SVError(fn, status, lib.sv_status_string(status).decode())


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ws(nbytes: int, device, ws: Optional[torch.Tensor]):
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError("workspace too small")
        return ws
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------


def attn_shape(q: torch.Tensor, k_cache: torch.Tensor) -> _AttnShape:
    B, R, Hq, D = q.shape
    _, Hkv, T_cap, _ = k_cache.shape
    return _AttnShape(B, R, Hq, Hkv, D, T_cap)


def verify_attn_workspace(B, R, Hq, Hkv, D, T_cap) -> int:
    s = _AttnShape(B, R, Hq, Hkv, D, T_cap)
    return int(lib.sv_verify_attn_workspace(ctypes.byref(s)))


ATTN_CACHE_READY = 1


def verify_attn(q, k_cache, v_cache, length, k_blk, v_blk, parent=None, scale=None, out=None, ws=None,
                stream=None, cache_ready=False):
    """q [B,R,Hq,D]; caches [B,Hkv,T_cap,D]; blocks [B,Hkv,R,D] (bf16); length [B] int32;
    parent None or [B,R] int32.  Returns out [B,R,Hq,D] bf16.  cache_ready: the
    kernel enqueued just before this call writes neither `length` nor the caches
    (sv_verify_attn_ex, SV_ATTN_CACHE_READY)."""
    s = attn_shape(q, k_cache)
    if scale is None:
        scale = q.shape[-1] ** -0.5
    if out is None:
        out = torch.empty_like(q)
    nbytes = int(lib.sv_verify_attn_workspace(ctypes.byref(s)))
    if ws is None and nbytes > 0:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)   # ticket words start at zero
    ws = _ws(nbytes, q.device, ws)
    bf = torch.bfloat16
    _check("sv_verify_attn_ex", lib.sv_verify_attn_ex(
        ctypes.byref(s), _ptr(q, bf, "q"), _ptr(k_cache, bf, "k_cache"), _ptr(v_cache, bf, "v_cache"),
        _ptr(length, torch.int32, "len"), _ptr(k_blk, bf, "k_blk"), _ptr(v_blk, bf, "v_blk"),
        _ptr(parent, torch.int32, "parent"), float(scale), _ptr(out, bf, "out"), _ptr(ws), nbytes,
        ATTN_CACHE_READY if cache_ready else 0, _stream(stream)))
    return out


KV_PAGE = 64   # positions per page of a paged cache (SV_KV_PAGE)


def verify_attn_paged(q, k_pool, v_pool, page_table, length, k_blk, v_blk, parent=None, scale=None, out=None,
                      ws=None, stream=None, cache_ready=False):
    """Paged cache: pools [num_pages,Hkv,64,D] bf16, page_table [B,max_pages] int32
    (position p of sequence b = row p % 64 of page page_table[b][p // 64]);
    other arguments as verify_attn.  Returns out [B,R,Hq,D] bf16."""
    B, R, Hq, D = q.shape
    num_pages, Hkv = k_pool.shape[0], k_pool.shape[1]
    max_pages = page_table.shape[1]
    s = _AttnShape(B, R, Hq, Hkv, D, max_pages * KV_PAGE)
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    nbytes = int(lib.sv_verify_attn_workspace(ctypes.byref(s)))
    if ws is None and nbytes > 0:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)   # ticket words start at zero
    ws = _ws(nbytes, q.device, ws)
    bf, i32 = torch.bfloat16, torch.int32
    _check("sv_verify_attn_paged", lib.sv_verify_attn_paged(
        ctypes.byref(s), _ptr(q, bf, "q"), _ptr(k_pool, bf, "k_pool"), _ptr(v_pool, bf, "v_pool"), num_pages,
        _ptr(page_table, i32, "page_table"), max_pages, _ptr(length, i32, "len"), _ptr(k_blk, bf, "k_blk"),
        _ptr(v_blk, bf, "v_blk"), _ptr(parent, i32, "parent"), float(scale), _ptr(out, bf, "out"), _ptr(ws), nbytes,
        ATTN_CACHE_READY if cache_ready else 0, _stream(stream)))
    return out


LM_WEIGHTS_READY = 1


def lm_head(hid, W, logits=None, stream=None, weights_ready=False):
    """hid [N,H] bf16; W [H,V] bf16 -> logits [N,V] fp32.  weights_ready: the
    kernel enqueued just before this call does not write W (sv_lm_head_ex,
    SV_LM_WEIGHTS_READY)."""
    N, H = hid.shape
    V = W.shape[1]
    if logits is None:
        logits = torch.empty(N, V, dtype=torch.float32, device=hid.device)
    _check("sv_lm_head_ex", lib.sv_lm_head_ex(_ptr(hid, torch.bfloat16, "hid"), _ptr(W, torch.bfloat16, "W"),
                                              _ptr(logits, torch.float32, "logits"), N, H, V,
                                              LM_WEIGHTS_READY if weights_ready else 0, _stream(stream)))
    return logits


ARGMAX_SLAB = 128   # vocab columns summarised by one argmax key (SV_ARGMAX_SLAB)


def lm_head_argmax(hid, W, logits=None, argmax=None, stream=None, weights_ready=False, write_logits=True):
    """hid [N,H] bf16; W [H,V] bf16 -> (logits [N,V] fp32 or None, argmax keys
    [N, ceil(V/128)] int64 holding the uint64 keys of sv_lm_head_argmax).
    write_logits=False passes NULL: only the keys are written."""
    N, H = hid.shape
    V = W.shape[1]
    if write_logits and logits is None:
        logits = torch.empty(N, V, dtype=torch.float32, device=hid.device)
    if not write_logits:
        logits = None
    S = (V + ARGMAX_SLAB - 1) // ARGMAX_SLAB
    if argmax is None:
        argmax = torch.empty(N, S, dtype=torch.int64, device=hid.device)
    nbytes = int(lib.sv_lm_head_argmax_bytes(N, V))
    if argmax.numel() * argmax.element_size() < nbytes:
        raise ValueError("argmax buffer too small")
    _check("sv_lm_head_argmax", lib.sv_lm_head_argmax(
        _ptr(hid, torch.bfloat16, "hid"), _ptr(W, torch.bfloat16, "W"), _ptr(logits, torch.float32, "logits"), N, H,
        V, _ptr(argmax, torch.int64, "argmax"), nbytes, LM_WEIGHTS_READY if weights_ready else 0, _stream(stream)))
    return logits, argmax


def accept_greedy_commit(argmax, tok, V, parent=None, n_acc=None, out_tok=None, path=None, k_cache=None,
                         v_cache=None, k_blk=None, v_blk=None, length=None, stream=None):
    """Greedy acceptance from lm_head_argmax's keys [B*R, S] and, when the
    caches are given (caches [L,B,Hkv,T_cap,D], blocks [L,B,Hkv,R,D] bf16,
    length [B] int32 updated in place), the KV commit, in one launch.
    Returns (n_acc [B], out_tok [B], path [B,R])."""
    B, R = tok.shape
    n_acc, out_tok, path = _accept_outputs(B, R, tok.device, n_acc, out_tok, path)
    bf, i32 = torch.bfloat16, torch.int32
    if k_cache is not None:
        L, _, Hkv, T_cap, D = k_cache.shape
    else:
        L = Hkv = T_cap = D = 0
    _check("sv_accept_greedy_commit", lib.sv_accept_greedy_commit(
        _ptr(argmax, torch.int64, "argmax"), _ptr(tok, i32, "tok"), _ptr(parent, i32, "parent"), B, R, V,
        _ptr(n_acc, i32), _ptr(out_tok, i32), _ptr(path, i32), _ptr(k_cache, bf, "k_cache"),
        _ptr(v_cache, bf, "v_cache"), _ptr(k_blk, bf, "k_blk"), _ptr(v_blk, bf, "v_blk"), L, Hkv, D, T_cap,
        _ptr(length, i32, "len"), _stream(stream)))
    return n_acc, out_tok, path


def accept_greedy_commit_paged(argmax, tok, V, k_pool, v_pool, page_table, k_blk, v_blk, length, parent=None,
                               n_acc=None, out_tok=None, path=None, stream=None):
    """accept_greedy_commit into paged caches: pools [L,num_pages,Hkv,64,D] bf16,
    page_table [B,max_pages] int32, blocks [L,B,Hkv,R,D] bf16, length [B]
    int32 (updated in place).  Returns (n_acc, out_tok, path)."""
    B, R = tok.shape
    n_acc, out_tok, path = _accept_outputs(B, R, tok.device, n_acc, out_tok, path)
    L, num_pages, Hkv, _, D = k_pool.shape
    bf, i32 = torch.bfloat16, torch.int32
    _check("sv_accept_greedy_commit_paged", lib.sv_accept_greedy_commit_paged(
        _ptr(argmax, torch.int64, "argmax"), _ptr(tok, i32, "tok"), _ptr(parent, i32, "parent"), B, R, V,
        _ptr(n_acc, i32), _ptr(out_tok, i32), _ptr(path, i32), _ptr(k_pool, bf, "k_pool"), _ptr(v_pool, bf, "v_pool"),
        num_pages, _ptr(page_table, i32, "page_table"), page_table.shape[1], _ptr(k_blk, bf, "k_blk"),
        _ptr(v_blk, bf, "v_blk"), L, Hkv, D, _ptr(length, i32, "len"), _stream(stream)))
    return n_acc, out_tok, path


def _accept_outputs(B, R, device, n_acc, out_tok, path):
    if n_acc is None:
        n_acc = torch.empty(B, dtype=torch.int32, device=device)
    if out_tok is None:
        out_tok = torch.empty(B, dtype=torch.int32, device=device)
    if path is None:
        path = torch.empty(B, R, dtype=torch.int32, device=device)
    return n_acc, out_tok, path


def accept_greedy(logits, tok, parent=None, n_acc=None, out_tok=None, path=None, ws=None, stream=None):
    """logits [B,R,V] fp32; tok [B,R] int32 -> (n_acc [B], out_tok [B], path [B,R])."""
    B, R, V = logits.shape
    n_acc, out_tok, path = _accept_outputs(B, R, logits.device, n_acc, out_tok, path)
    nbytes = int(lib.sv_accept_greedy_workspace(B, R, V))
    ws = _ws(nbytes, logits.device, ws)
    i32 = torch.int32
    _check("sv_accept_greedy", lib.sv_accept_greedy(
        _ptr(logits, torch.float32, "logits"), _ptr(tok, i32, "tok"), _ptr(parent, i32, "parent"), B, R, V,
        _ptr(n_acc, i32), _ptr(out_tok, i32), _ptr(path, i32), _ptr(ws), nbytes, _stream(stream)))
    return n_acc, out_tok, path


def accept_greedy_relaxed(logits, tok, parent=None, delta=0.0, n_acc=None, out_tok=None, path=None, ws=None,
                          stream=None):
    """Lossy Delta-logit acceptance: as accept_greedy, but a draft passes when
    its parent row's top-1 logit exceeds its logit by at most delta."""
    B, R, V = logits.shape
    n_acc, out_tok, path = _accept_outputs(B, R, logits.device, n_acc, out_tok, path)
    nbytes = int(lib.sv_accept_greedy_relaxed_workspace(B, R, V))
    ws = _ws(nbytes, logits.device, ws)
    i32 = torch.int32
    _check("sv_accept_greedy_relaxed", lib.sv_accept_greedy_relaxed(
        _ptr(logits, torch.float32, "logits"), _ptr(tok, i32, "tok"), _ptr(parent, i32, "parent"), B, R, V,
        float(delta), _ptr(n_acc, i32), _ptr(out_tok, i32), _ptr(path, i32), _ptr(ws), nbytes, _stream(stream)))
    return n_acc, out_tok, path


def _check_sample_shapes(logits, q, tok, parent):
    """q holds one draft distribution per chain position (R - 1 rows) or per
    tree node (R rows); the C ABI cannot see its row count, so it is checked
    here."""
    B, R, _ = logits.shape
    rq = R if parent is not None else R - 1
    if q.dim() != 3 or q.shape[0] != B or q.shape[1] != rq:
        raise ValueError(f"q must be [B, {rq}, Vq] for a {'tree' if parent is not None else 'chain'} of R = {R} "
                         f"rows, got {tuple(q.shape)}")
    if tuple(tok.shape) != (B, R):
        raise ValueError(f"tok must be [B, R] = [{B}, {R}], got {tuple(tok.shape)}")
    if parent is not None and tuple(parent.shape) != (B, R):
        raise ValueError(f"parent must be [B, R] = [{B}, {R}], got {tuple(parent.shape)}")


def accept_sample(logits, q, tok, parent=None, temperature=1.0, seed=0, step=0, uniforms=None, n_acc=None,
                  out_tok=None, path=None, ws=None, stream=None):
    """logits [B,R,V] fp32; q [B,R-1 (chain) or R (tree),Vq] fp32; tok [B,R] int32;
    uniforms None (Philox) or [B,R,2] fp32."""
    _check_sample_shapes(logits, q, tok, parent)
    B, R, V = logits.shape
    Vq = q.shape[-1]
    n_acc, out_tok, path = _accept_outputs(B, R, logits.device, n_acc, out_tok, path)
    nbytes = int(lib.sv_accept_sample_workspace(B, R, V))
    ws = _ws(nbytes, logits.device, ws)
    i32, f32 = torch.int32, torch.float32
    _check("sv_accept_sample", lib.sv_accept_sample(
        _ptr(logits, f32, "logits"), _ptr(q, f32, "q"), Vq, _ptr(tok, i32, "tok"), _ptr(parent, i32, "parent"),
        B, R, V, float(temperature), int(seed) & (2 ** 64 - 1), int(step) & (2 ** 64 - 1),
        _ptr(uniforms, f32, "uniforms"), _ptr(n_acc, i32), _ptr(out_tok, i32), _ptr(path, i32), _ptr(ws), nbytes,
        _stream(stream)))
    return n_acc, out_tok, path


def accept_sample_noalloc(logits, q, tok, parent=None, temperature=1.0, seed=0, step=0, uniforms=None, n_acc=None,
                          out_tok=None, path=None, stream=None):
    """accept_sample for callers that cannot allocate device memory: the
    library's fixed scratch array replaces the workspace (B*R <= 8192; calls
    overlapping on the GPU race on it)."""
    _check_sample_shapes(logits, q, tok, parent)
    B, R, V = logits.shape
    Vq = q.shape[-1]
    n_acc, out_tok, path = _accept_outputs(B, R, logits.device, n_acc, out_tok, path)
    i32, f32 = torch.int32, torch.float32
    _check("sv_accept_sample_noalloc", lib.sv_accept_sample_noalloc(
        _ptr(logits, f32, "logits"), _ptr(q, f32, "q"), Vq, _ptr(tok, i32, "tok"), _ptr(parent, i32, "parent"),
        B, R, V, float(temperature), int(seed) & (2 ** 64 - 1), int(step) & (2 ** 64 - 1),
        _ptr(uniforms, f32, "uniforms"), _ptr(n_acc, i32), _ptr(out_tok, i32), _ptr(path, i32), _stream(stream)))
    return n_acc, out_tok, path


def kv_commit(k_cache, v_cache, k_blk, v_blk, path, n_acc, length, stream=None):
    """caches [L,B,Hkv,T_cap,D]; blocks [L,B,Hkv,R,D] (bf16); path [B,R], n_acc [B], length [B] int32
    (length updated in place)."""
    L, B, Hkv, T_cap, D = k_cache.shape
    R = k_blk.shape[3]
    bf, i32 = torch.bfloat16, torch.int32
    _check("sv_kv_commit", lib.sv_kv_commit(
        _ptr(k_cache, bf, "k_cache"), _ptr(v_cache, bf, "v_cache"), _ptr(k_blk, bf, "k_blk"),
        _ptr(v_blk, bf, "v_blk"), L, B, Hkv, D, T_cap, R, _ptr(path, i32, "path"), _ptr(n_acc, i32, "n_acc"),
        _ptr(length, i32, "len"), _stream(stream)))


def kv_commit_paged(k_pool, v_pool, page_table, k_blk, v_blk, path, n_acc, length, stream=None):
    """pools [L,num_pages,Hkv,64,D]; page_table [B,max_pages]; blocks [L,B,Hkv,R,D] (bf16);
    path [B,R], n_acc [B], length [B] int32 (length updated in place)."""
    L, num_pages, Hkv, _, D = k_pool.shape
    B, R = k_blk.shape[1], k_blk.shape[3]
    bf, i32 = torch.bfloat16, torch.int32
    _check("sv_kv_commit_paged", lib.sv_kv_commit_paged(
        _ptr(k_pool, bf, "k_pool"), _ptr(v_pool, bf, "v_pool"), num_pages, _ptr(page_table, i32, "page_table"),
        page_table.shape[1], _ptr(k_blk, bf, "k_blk"), _ptr(v_blk, bf, "v_blk"), L, B, Hkv, D, R,
        _ptr(path, i32, "path"), _ptr(n_acc, i32, "n_acc"), _ptr(length, i32, "len"), _stream(stream)))


def copy(dst: torch.Tensor, src: torch.Tensor, stream=None) -> torch.Tensor:
    """dst <- src (same byte count, contiguous) by sv_copy: each side a CUDA
    tensor or a pinned CPU tensor; the copy is a kernel on the stream."""
    for name, t in (("dst", dst), ("src", src)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda and not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst and src must hold the same number of bytes")
    _check("sv_copy", lib.sv_copy(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), nbytes,
                                  _stream(stream)))
    return dst


def get_device_error(stream=None) -> int:
    word = ctypes.c_uint32(0)
    st = lib.sv_get_device_error(ctypes.byref(word), _stream(stream))
    if st not in (0, 6):
        _check("sv_get_device_error", st)
    return int(word.value)


def diag_exp(x: torch.Tensor, stream=None) -> torch.Tensor:
    y = torch.empty_like(x)
    _check("sv_diag_exp", lib.sv_diag_exp(_ptr(x, torch.float32), _ptr(y, torch.float32), x.numel(),
                                          _stream(stream)))
    return y


def diag_div(a: torch.Tensor, b: torch.Tensor, stream=None) -> torch.Tensor:
    """Elementwise a / b (float32, same shape) through the acceptance's division."""
    if a.shape != b.shape:
        raise ValueError("a and b differ in shape")
    q = torch.empty_like(a)
    _check("sv_diag_div", lib.sv_diag_div(_ptr(a, torch.float32), _ptr(b, torch.float32), _ptr(q, torch.float32),
                                          a.numel(), _stream(stream)))
    return q


def diag_philox(ctr: torch.Tensor, key: torch.Tensor, stream=None) -> torch.Tensor:
    """ctr [n,4] int32 (bit patterns), key [n,2] int32 -> [n,4] int32."""
    out = torch.empty_like(ctr)
    _check("sv_diag_philox", lib.sv_diag_philox(_ptr(ctr, torch.int32), _ptr(key, torch.int32),
                                                _ptr(out, torch.int32), ctr.shape[0], _stream(stream)))
    return out


def diag_canon(x: torch.Tensor, u: torch.Tensor, stream=None):
    """x [m,n] fp32, u [m] fp32 -> (sums [m] fp32, draws [m] int32)."""
    m, n = x.shape
    sums = torch.empty(m, dtype=torch.float32, device=x.device)
    draws = torch.empty(m, dtype=torch.int32, device=x.device)
    _check("sv_diag_canon", lib.sv_diag_canon(_ptr(x, torch.float32), n, m, _ptr(u, torch.float32),
                                              _ptr(sums), _ptr(draws), _stream(stream)))
    return sums, draws
