"""CPU oracle for the speculative-decoding block-verification step.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers; the product path never
imports this package.  It shares no code with the CUDA library: the arithmetic
lives in ``sv_oracle.c`` (plain C, built with ``-ffp-contract=off``); this
module only compiles it and marshals numpy arrays.

bf16 tensors cross this boundary as ``numpy.uint16`` arrays holding the raw
bf16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sv_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if the compiler has it)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", _SRC, "-o", _LIB_PATH + ".tmp"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, u64, f32, f64 = ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_double
            L.orc_num_threads.restype = i32
            L.orc_philox4x32_10.argtypes = [P, P, P]
            L.orc_uniform24.argtypes = [ctypes.c_uint32]
            L.orc_uniform24.restype = f32
            L.orc_exp.argtypes = [f32]
            L.orc_exp.restype = f32
            L.orc_exp_array.argtypes = [P, P, ctypes.c_long]
            L.orc_tree_sample_batch.argtypes = [P, i32, P, ctypes.c_long, P]
            L.orc_canon_sum.argtypes = [P, i32]
            L.orc_canon_sum.restype = f32
            L.orc_tree_sample.argtypes = [P, i32, f32]
            L.orc_tree_sample.restype = i32
            L.orc_softmax.argtypes = [P, i32, f32, P]
            L.orc_accept_greedy.argtypes = [P, P, P, i32, i32, i32, P, P, P]
            L.orc_accept_greedy.restype = i32
            L.orc_accept_greedy_relaxed.argtypes = [P, P, P, i32, i32, i32, f32, P, P, P]
            L.orc_accept_greedy_relaxed.restype = i32
            L.orc_accept_sample.argtypes = [P, P, i32, P, P, i32, i32, i32, f32, u64, u64, P, P, P, P]
            L.orc_accept_sample.restype = i32
            L.orc_kv_commit.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, P, P, P]
            L.orc_kv_commit.restype = i32
            L.orc_verify_attn.argtypes = [i32, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, f64, P]
            L.orc_verify_attn.restype = i32
            L.orc_lm_head.argtypes = [P, P, i32, i32, i32, i32, i32, P]
            L.orc_lm_head.restype = i32
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


class OracleError(RuntimeError):
    pass


def num_threads() -> int:
    return lib().orc_num_threads()


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32).reshape(4).copy()
    k = np.asarray(key, dtype=np.uint32).reshape(2).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def uniform24(w: int) -> float:
    return lib().orc_uniform24(int(w) & 0xFFFFFFFF)


def exp32(x: float) -> float:
    return lib().orc_exp(float(x))


def exp32_array(xs):
    x = _c(xs, np.float32)
    y = np.empty_like(x)
    lib().orc_exp_array(_p(x), _p(y), x.size)
    return y


def canon_sum(x) -> float:
    x = _c(x, np.float32)
    return lib().orc_canon_sum(_p(x), x.size)


def tree_sample(x, u: float) -> int:
    x = _c(x, np.float32)
    return lib().orc_tree_sample(_p(x), x.size, float(u))


def tree_sample_batch(x, us):
    x = _c(x, np.float32)
    us = _c(us, np.float32)
    out = np.empty(us.size, np.int32)
    lib().orc_tree_sample_batch(_p(x), x.size, _p(us), us.size, _p(out))
    return out


def softmax(l, T: float = 1.0):
    l = _c(l, np.float32)
    p = np.empty_like(l)
    lib().orc_softmax(_p(l), l.size, float(T), _p(p))
    return p


def accept_greedy(logits, tok, parent=None):
    """logits [B, R, V] float32; tok [B, R] int32; parent None or [B, R]."""
    logits = _c(logits, np.float32)
    B, R, V = logits.shape
    tok = _c(tok, np.int32)
    parent = _c(parent, np.int32)
    n_acc = np.zeros(B, np.int32)
    out_tok = np.zeros(B, np.int32)
    path = np.zeros((B, R), np.int32)
    rc = lib().orc_accept_greedy(_p(logits), _p(tok), _p(parent), B, R, V, _p(n_acc), _p(out_tok), _p(path))
    if rc != 0:
        raise OracleError("orc_accept_greedy rejected its inputs")
    return n_acc, out_tok, path


def accept_greedy_relaxed(logits, tok, parent=None, delta=0.0):
    """Lossy Delta-logit acceptance ([SCS] sec. 7.2): draft passes iff
    top1 logit - draft logit <= delta (float32).  Shapes as accept_greedy."""
    logits = _c(logits, np.float32)
    B, R, V = logits.shape
    tok = _c(tok, np.int32)
    parent = _c(parent, np.int32)
    n_acc = np.zeros(B, np.int32)
    out_tok = np.zeros(B, np.int32)
    path = np.zeros((B, R), np.int32)
    rc = lib().orc_accept_greedy_relaxed(_p(logits), _p(tok), _p(parent), B, R, V, float(delta), _p(n_acc),
                                         _p(out_tok), _p(path))
    if rc != 0:
        raise OracleError("orc_accept_greedy_relaxed rejected its inputs")
    return n_acc, out_tok, path


def accept_sample(logits, q, tok, parent=None, temperature=1.0, seed=0, step=0, uniforms=None):
    """logits [B, R, V]; q [B, R-1 (chain) or R (tree), Vq]; uniforms None or [B, R, 2]."""
    logits = _c(logits, np.float32)
    B, R, V = logits.shape
    q = _c(q, np.float32)
    Vq = q.shape[-1]
    tok = _c(tok, np.int32)
    parent = _c(parent, np.int32)
    uniforms = _c(uniforms, np.float32)
    n_acc = np.zeros(B, np.int32)
    out_tok = np.zeros(B, np.int32)
    path = np.zeros((B, R), np.int32)
    rc = lib().orc_accept_sample(_p(logits), _p(q), Vq, _p(tok), _p(parent), B, R, V, float(temperature),
                                 int(seed) & (2**64 - 1), int(step) & (2**64 - 1), _p(uniforms),
                                 _p(n_acc), _p(out_tok), _p(path))
    if rc != 0:
        raise OracleError("orc_accept_sample rejected its inputs")
    return n_acc, out_tok, path


def kv_commit(k_cache, v_cache, k_blk, v_blk, path, n_acc, length):
    """In place on copies: returns (k_cache, v_cache, len) after the commit.
    cache [L, B, Hkv, T_cap, D] uint16; block [L, B, Hkv, R, D] uint16."""
    kc = _c(k_cache, np.uint16).copy()
    vc = _c(v_cache, np.uint16).copy()
    kb = _c(k_blk, np.uint16)
    vb = _c(v_blk, np.uint16)
    L, B, Hkv, T_cap, D = kc.shape
    R = kb.shape[3]
    path = _c(path, np.int32)
    n_acc = _c(n_acc, np.int32)
    ln = _c(length, np.int32).copy()
    rc = lib().orc_kv_commit(_p(kc), _p(vc), _p(kb), _p(vb), L, B, Hkv, D, T_cap, R, _p(path), _p(n_acc), _p(ln))
    if rc != 0:
        raise OracleError("orc_kv_commit rejected its inputs")
    return kc, vc, ln


def gather_pages(pool, page_table, page=64):
    """The contiguous cache a paged one stands for ([MINI] implementation
    architecture: KV in a block tensor addressed through the block table):
    pool [..., P, Hkv, page, D], page_table [B, max_pages] ->
    [..., B, Hkv, max_pages * page, D], where position p of sequence b is row
    p % page of page page_table[b][p // page].  A plain re-layout (numpy
    indexing), no arithmetic."""
    pool = np.asarray(pool)
    tab = np.asarray(page_table, np.int64)
    B, M = tab.shape
    g = pool[..., tab, :, :, :]                       # [..., B, M, Hkv, page, D]
    g = np.moveaxis(g, -3, -4)                        # [..., B, Hkv, M, page, D]
    return np.ascontiguousarray(g.reshape(g.shape[:-3] + (M * page, g.shape[-1])))


def scatter_pages(pool, page_table, cache, page=64):
    """Inverse of gather_pages for the pages the table names (each named
    once): returns a copy of pool with those pages taken from cache."""
    out = np.array(pool, copy=True)
    tab = np.asarray(page_table, np.int64)
    B, M = tab.shape
    c = np.asarray(cache)
    c = c.reshape(c.shape[:-2] + (M, page, c.shape[-1]))   # [..., B, Hkv, M, page, D]
    c = np.moveaxis(c, -3, -4)                              # [..., B, M, Hkv, page, D]
    out[..., tab, :, :, :] = c
    return out


def verify_attn(q, k_cache, v_cache, length, k_blk, v_blk, parent=None, scale=None):
    """q [B, R, Hq, D] uint16; cache [B, Hkv, T_cap, D]; block [B, Hkv, R, D];
    returns float64 [B, R, Hq, D]."""
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    kb = _c(k_blk, np.uint16)
    vb = _c(v_blk, np.uint16)
    B, R, Hq, D = q.shape
    Hkv, T_cap = kc.shape[1], kc.shape[2]
    ln = _c(length, np.int32)
    parent = _c(parent, np.int32)
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((B, R, Hq, D), np.float64)
    rc = lib().orc_verify_attn(B, R, Hq, Hkv, D, T_cap, _p(q), _p(kc), _p(vc), _p(ln), _p(kb), _p(vb),
                               _p(parent), float(scale), _p(out))
    if rc != 0:
        raise OracleError("orc_verify_attn rejected its inputs")
    return out


def lm_head(hid, W, v0=0, v1=None):
    """hid [N, H] uint16; W [H, V] uint16; returns float64 [N, v1 - v0]."""
    hid = _c(hid, np.uint16)
    W = _c(W, np.uint16)
    N, H = hid.shape
    V = W.shape[1]
    if v1 is None:
        v1 = V
    out = np.zeros((N, v1 - v0), np.float64)
    rc = lib().orc_lm_head(_p(hid), _p(W), N, H, V, int(v0), int(v1), _p(out))
    if rc != 0:
        raise OracleError("orc_lm_head rejected its inputs")
    return out
