"""Pins for the oracle's verify attention, LM head and KV commit.

Attention ([SpecDec-Context-Scaling guide, sec. 3]; [wmrh.cn tutorial,
sec. 3.2]; [SubSpec summary, sec. 4.2]): closed forms (one visible key gives
its value; equal keys give the mean of the visible values), the chain mask
equals the tree mask of a path, and an independent library routine
(torch scaled_dot_product_attention in float64 with an explicit mask).

LM head: one-hot hidden rows reproduce rows of W exactly; a float64 numpy
matmul and an exact rational sum agree.

KV commit ([SpecDec-Context-Scaling guide, sec. 3.2]; [mini-infer Phase 11,
hidden KV position bug]): hand-built golden cases; the length invariant; the
accepted rows land bit for bit at t..t+m and nothing else changes.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_sv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(x: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(x)


def _rand_attn(B, R, Hq, Hkv, D, T_cap, t, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    return (mk(B, R, Hq, D), mk(B, Hkv, T_cap, D), mk(B, Hkv, T_cap, D), mk(B, Hkv, R, D), mk(B, Hkv, R, D),
            np.array(t, np.int32))


def _sdpa_reference(q, kc, vc, kb, vb, t, parent, scale):
    B, R, Hq, D = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    out = torch.zeros(B, R, Hq, D, dtype=torch.float64)
    for b in range(B):
        tb = int(t[b])
        keys = torch.cat([kc[b, :, :tb], kb[b]], dim=1).double()       # [Hkv, tb+R, D]
        vals = torch.cat([vc[b, :, :tb], vb[b]], dim=1).double()
        mask = torch.zeros(R, tb + R, dtype=torch.bool)
        mask[:, :tb] = True
        for j in range(R):
            if parent is None:
                mask[j, tb:tb + j + 1] = True
            else:
                i = j
                while i >= 0:
                    mask[j, tb + i] = True
                    i = int(parent[b, i])
        qq = q[b].double().permute(1, 0, 2)                                 # [Hq, R, D]
        kk = keys.repeat_interleave(G, dim=0)
        vv = vals.repeat_interleave(G, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
        out[b] = o.permute(1, 0, 2)
    return out.numpy()


@pytest.mark.parametrize("tree", [False, True])
def test_attn_matches_sdpa_float64(tree):
    B, R, Hq, Hkv, D, T_cap = 3, 5, 6, 2, 16, 40
    t = [0, 17, 33]
    q, kc, vc, kb, vb, ln = _rand_attn(B, R, Hq, Hkv, D, T_cap, t, 21)
    parent = None
    if tree:
        parent = np.array([[-1, 0, 0, 1, 1], [-1, 0, 1, 2, 3], [-1, 0, 0, 0, 2]], np.int32)
    got = oracle.verify_attn(_bits(q), _bits(kc), _bits(vc), ln, _bits(kb), _bits(vb), parent, 0.3)
    ref = _sdpa_reference(q, kc, vc, kb, vb, ln, parent, 0.3)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_attn_single_visible_key_returns_its_value():
    # R = 1, t = 0: the pending token sees only itself.
    q, kc, vc, kb, vb, _ = _rand_attn(2, 1, 4, 2, 8, 8, [0, 0], 22)
    got = oracle.verify_attn(_bits(q), _bits(kc), _bits(vc), np.array([0, 0], np.int32), _bits(kb), _bits(vb))
    G = 2
    for b in range(2):
        for h in range(4):
            assert np.array_equal(got[b, 0, h], vb[b, h // G, 0].double().numpy())


def test_attn_equal_keys_give_mean_of_visible_values():
    B, R, Hq, Hkv, D, T_cap, t = 1, 4, 2, 1, 8, 16, 6
    q, kc, vc, kb, vb, _ = _rand_attn(B, R, Hq, Hkv, D, T_cap, [t], 23)
    key = torch.randn(D).to(torch.bfloat16)
    kc[:] = key
    kb[:] = key
    got = oracle.verify_attn(_bits(q), _bits(kc), _bits(vc), np.array([t], np.int32), _bits(kb), _bits(vb))
    for j in range(R):
        vis = torch.cat([vc[0, 0, :t], vb[0, 0, :j + 1]]).double()
        assert np.allclose(got[0, j, 0], vis.mean(0).numpy(), atol=1e-12)


def test_attn_chain_equals_path_tree():
    B, R, Hq, Hkv, D, T_cap = 2, 6, 4, 2, 32, 64
    q, kc, vc, kb, vb, ln = _rand_attn(B, R, Hq, Hkv, D, T_cap, [50, 9], 24)
    parent = np.tile(np.arange(-1, R - 1, dtype=np.int32), (B, 1))
    a = oracle.verify_attn(_bits(q), _bits(kc), _bits(vc), ln, _bits(kb), _bits(vb))
    b = oracle.verify_attn(_bits(q), _bits(kc), _bits(vc), ln, _bits(kb), _bits(vb), parent)
    assert np.array_equal(a, b)


def test_attn_rejects_bad_tree_and_length():
    q, kc, vc, kb, vb, ln = _rand_attn(1, 3, 2, 1, 8, 8, [4], 25)
    with pytest.raises(oracle.OracleError):
        oracle.verify_attn(_bits(q), _bits(kc), _bits(vc), ln, _bits(kb), _bits(vb), np.array([[-1, 2, 0]], np.int32))
    with pytest.raises(oracle.OracleError):
        oracle.verify_attn(_bits(q), _bits(kc), _bits(vc), np.array([9], np.int32), _bits(kb), _bits(vb))


# ----------------------------------------------------------------------------
# LM head
# ----------------------------------------------------------------------------

def test_lm_head_one_hot_rows_copy_w():
    H, V = 24, 50
    W = (torch.randn(H, V) * 0.02).to(torch.bfloat16)
    hid = torch.zeros(3, H, dtype=torch.bfloat16)
    for r, h in enumerate((0, 7, 23)):
        hid[r, h] = 1.0
    got = oracle.lm_head(_bits(hid), _bits(W))
    for r, h in enumerate((0, 7, 23)):
        assert np.array_equal(got[r], W[h].double().numpy())


def test_lm_head_matches_numpy_and_exact_sum():
    N, H, V = 5, 96, 70
    hid = torch.randn(N, H).to(torch.bfloat16)
    W = (torch.randn(H, V) * 0.02).to(torch.bfloat16)
    got = oracle.lm_head(_bits(hid), _bits(W))
    ref = hid.double().numpy() @ W.double().numpy()
    assert np.max(np.abs(got - ref)) < 1e-12
    hf = [[Fraction(float(x)) for x in row] for row in hid.float().numpy()]
    wf = [[Fraction(float(x)) for x in row] for row in W.float().numpy()]
    for r in range(N):
        for v in range(0, V, 13):
            exact = sum(hf[r][h] * wf[h][v] for h in range(H))
            assert abs(float(exact) - got[r, v]) <= 1e-15 * (1 + abs(float(exact)))
    part = oracle.lm_head(_bits(hid), _bits(W), 11, 37)
    assert np.array_equal(part, got[:, 11:37])


# ----------------------------------------------------------------------------
# KV commit
# ----------------------------------------------------------------------------

def test_commit_golden():
    g = json.load(open(os.path.join(GOLDEN, "commit.json")))
    T_cap, R = g["T_cap"], g["R"]
    for case in g["cases"]:
        kc = np.array(case["cache_before"], np.uint16).reshape(1, 1, 1, T_cap, 1)
        kb = np.array(case["block"], np.uint16).reshape(1, 1, 1, R, 1)
        vc = kc + 1000
        vb = kb + 1000
        path = np.array([case["path"]], np.int32)
        k2, v2, ln = oracle.kv_commit(kc, vc, kb, vb, path, np.array([case["n_acc"]], np.int32),
                                      np.array([case["t"]], np.int32))
        assert k2.reshape(-1).tolist() == case["cache_after"], case["why"]
        assert (v2.reshape(-1) - 1000).tolist() == case["cache_after"], case["why"]
        assert int(ln[0]) == case["len_after"], case["why"]


def test_commit_invariant_random():
    rng = np.random.default_rng(31)
    L, B, Hkv, T_cap, D, R = 3, 5, 2, 48, 16, 9
    kc = rng.integers(0, 65535, size=(L, B, Hkv, T_cap, D), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(L, B, Hkv, T_cap, D), dtype=np.uint16)
    kb = rng.integers(0, 65535, size=(L, B, Hkv, R, D), dtype=np.uint16)
    vb = rng.integers(0, 65535, size=(L, B, Hkv, R, D), dtype=np.uint16)
    t = rng.integers(0, T_cap - R, size=B).astype(np.int32)
    n_acc = rng.integers(0, R, size=B).astype(np.int32)
    path = np.full((B, R), -1, np.int32)
    for b in range(B):
        # a root-to-node path of a tree: increasing node ids starting at 0
        nodes = np.sort(rng.choice(np.arange(1, R), size=n_acc[b], replace=False))
        path[b, :n_acc[b] + 1] = np.concatenate([[0], nodes])
    k2, v2, ln = oracle.kv_commit(kc, vc, kb, vb, path, n_acc, t)
    assert np.array_equal(ln, t + n_acc + 1)
    for b in range(B):
        m = n_acc[b]
        for i in range(m + 1):
            assert np.array_equal(k2[:, b, :, t[b] + i], kb[:, b, :, path[b, i]])
            assert np.array_equal(v2[:, b, :, t[b] + i], vb[:, b, :, path[b, i]])
        keep = np.ones(T_cap, bool)
        keep[t[b]:t[b] + m + 1] = False
        assert np.array_equal(k2[:, b, :, keep], kc[:, b, :, keep])
        assert np.array_equal(v2[:, b, :, keep], vc[:, b, :, keep])


def test_commit_capacity_overflow_is_an_error():
    kc = np.zeros((1, 1, 1, 8, 4), np.uint16)
    kb = np.zeros((1, 1, 1, 4, 4), np.uint16)
    with pytest.raises(oracle.OracleError):
        oracle.kv_commit(kc, kc, kb, kb, np.array([[0, 1, 2, 3]], np.int32), np.array([3], np.int32),
                         np.array([5], np.int32))


def test_gather_and_scatter_pages_brute_force():
    """The paged cache's re-layout against its definition ([mini-infer Phase 11],
    block tensor and block table): position p of sequence b is row p % page of
    page table[b][p // page], checked element by element on a tiny pool."""
    rng = np.random.default_rng(12)
    L, P, H, page, D, B, M = 2, 9, 3, 4, 5, 2, 3
    pool = rng.integers(0, 60000, size=(L, P, H, page, D)).astype(np.uint16)
    table = np.array([[7, 0, 4], [2, 8, 5]], np.int32)
    c = oracle.gather_pages(pool, table, page=page)
    assert c.shape == (L, B, H, M * page, D)
    for l in range(L):
        for b in range(B):
            for h in range(H):
                for p in range(M * page):
                    assert np.array_equal(c[l, b, h, p], pool[l, table[b, p // page], h, p % page])
    # scatter writes back exactly the named pages
    c2 = c.copy()
    c2[:, 1, :, 5] = 1                                   # sequence 1, position 5: page 8, row 1
    back = oracle.scatter_pages(pool, table, c2, page=page)
    changed = np.argwhere(back != pool)
    assert set(map(tuple, changed[:, [1, 3]])) <= {(8, 1)}
    assert np.array_equal(back[:, 8, :, 1], np.ones_like(back[:, 8, :, 1]))
    for unnamed in (1, 3, 6):
        assert np.array_equal(back[:, unnamed], pool[:, unnamed])
