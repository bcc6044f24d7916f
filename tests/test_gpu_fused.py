"""GPU parity of the greedy argmax fused into the LM head
(sv_lm_head_argmax) and of greedy acceptance with the KV commit in one launch
(sv_accept_greedy_commit).

The hidden rows and weights are drawn so that every logit is exact in float32
whatever the summation order (small integers times a power of two, bounded
sums).  The oracle's LM head then yields the very logits the kernel forms, and
the oracle's greedy acceptance and commit on them are the expected result,
bit for bit -- no oracle input comes from the GPU.  Integer-valued logits also
tie often, inside a 128-column slab and across slab edges, so the lowest-index
rule is exercised without planting; the tests plant further ties at slab
edges by duplicating weight columns."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_sv_gb300 import synth

from _helpers import assert_same, bits

pytestmark = pytest.mark.gpu
SLAB = 128


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_sv_gb300 import binding
    return binding


def _bf16(a: np.ndarray) -> torch.Tensor:
    """float32 values exactly representable in bf16 -> bf16 tensor."""
    t = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.from_numpy(a.astype(np.float32)))
    return t


def _exact_lm(N, H, V, seed, tie_cols=()):
    """hid in {-2..2}, W = k * 2^-6 with |k| <= 64: every partial sum is a
    multiple of 2^-6 below 2^17 in magnitude, exact in float32.  Columns in
    tie_cols (c, c') copy column c into c'."""
    rng = np.random.default_rng(seed)
    hid = rng.integers(-2, 3, size=(N, H)).astype(np.float32)
    W = (rng.integers(-64, 65, size=(H, V)) * 2.0 ** -6).astype(np.float32)
    for c, c2 in tie_cols:
        W[:, c2] = W[:, c]
    assert 2 * 64 * 2.0 ** -6 * H < 2 ** 17
    return _bf16(hid), _bf16(W)


def _oracle_logits(hid, W):
    return oracle.lm_head(bits(hid), bits(W)).astype(np.float32)


def _keys_ref(logits: np.ndarray) -> np.ndarray:
    """The argmax keys by their definition: per row and 128-column slab the
    largest (okey(x) << 32 | ~col), okey(NaN) = 0, -0 as +0."""
    N, V = logits.shape
    x = (logits + np.float32(0.0)).astype(np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    ok = np.where(b & 0x80000000, ~b & 0xFFFFFFFF, b | 0x80000000)
    ok = np.where(np.isnan(logits), 0, ok).astype(np.uint64)
    col = np.arange(V, dtype=np.uint64)
    keys = (ok << np.uint64(32)) | (~col & np.uint64(0xFFFFFFFF))
    S = -(-V // SLAB)
    pad = np.zeros((N, S * SLAB), np.uint64)
    pad[:, :V] = keys
    return pad.reshape(N, S, SLAB).max(-1)


@pytest.mark.parametrize("N,H,V", [(1, 256, 151936), (5, 512, 151936), (9, 256, 152064), (16, 256, 4000),
                                   (17, 256, 30000), (65, 128, 152064), (144, 128, 152064), (40, 64, 1000)])
def test_lm_head_argmax_keys_and_logits(sv, N, H, V):
    """Both LM-head kernels (<= 16 rows: mma.sync; more: tcgen05): the logits
    equal the oracle's exactly (exact arithmetic), the keys equal their
    definition over those logits, with and without the logits written."""
    hid, W = _exact_lm(N, H, V, seed=N * 7 + H, tie_cols=[(5, SLAB), (SLAB - 1, 3 * SLAB), (2 * SLAB, 2 * SLAB - 1)])
    ref = _oracle_logits(hid, W)
    lg, keys = sv.lm_head_argmax(hid.cuda(), W.cuda())
    assert np.array_equal(lg.cpu().numpy(), ref)
    want = _keys_ref(ref)
    assert np.array_equal(keys.cpu().numpy().view(np.uint64), want)
    none, keys2 = sv.lm_head_argmax(hid.cuda(), W.cuda(), write_logits=False)
    assert none is None and torch.equal(keys, keys2)
    # the logits equal those of the plain LM head bit for bit
    assert torch.equal(sv.lm_head(hid.cuda(), W.cuda()), lg)
    assert sv.get_device_error() == 0


def _caches(L, B, Hkv, T_cap, R, seed):
    rng = np.random.default_rng(seed)
    kc = rng.integers(0, 65535, size=(L, B, Hkv, T_cap, 128), dtype=np.uint16)
    vc = rng.integers(0, 65535, size=(L, B, Hkv, T_cap, 128), dtype=np.uint16)
    kb = rng.integers(0, 65535, size=(L, B, Hkv, R, 128), dtype=np.uint16)
    vb = rng.integers(0, 65535, size=(L, B, Hkv, R, 128), dtype=np.uint16)
    return kc, vc, kb, vb


def _t(a):
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).cuda()


def _run_fused(sv, hid, W, tok, parent, kc, vc, kb, vb, t):
    V = W.shape[1]
    kct, vct = _t(kc), _t(vc)
    ln = torch.from_numpy(t.copy()).cuda()
    _, keys = sv.lm_head_argmax(hid.cuda(), W.cuda(), write_logits=False)
    pt = None if parent is None else torch.from_numpy(parent).cuda()
    out = sv.accept_greedy_commit(keys, torch.from_numpy(tok).cuda(), V, parent=pt, k_cache=kct, v_cache=vct,
                                  k_blk=_t(kb), v_blk=_t(vb), length=ln)
    return out, bits(kct), bits(vct), ln.cpu().numpy()


@pytest.mark.parametrize("B,R,H,V,L,Hkv,rate", [(1, 5, 512, 151936, 28, 2, 0.52), (16, 9, 128, 152064, 4, 4, 0.55),
                                                 (3, 4, 256, 30000, 2, 2, 0.9), (2, 1, 128, 4000, 3, 1, 0.5)])
def test_fused_chain_vs_oracle(sv, B, R, H, V, L, Hkv, rate):
    hid, W = _exact_lm(B * R, H, V, seed=B * 31 + R, tie_cols=[(7, SLAB + 7), (SLAB - 1, SLAB)])
    logits = _oracle_logits(hid, W).reshape(B, R, V)
    g = logits.argmax(-1)
    tok = synth.plant_chain_drafts(g, rate, V, seed=B + R)
    T_cap = 256
    t = np.random.default_rng(B).integers(0, T_cap - R + 1, size=B).astype(np.int32)
    kc, vc, kb, vb = _caches(L, B, Hkv, T_cap, R, seed=R)
    exp = oracle.accept_greedy(logits, tok)
    k_ref, v_ref, ln_ref = oracle.kv_commit(kc, vc, kb, vb, exp[2], exp[0], t)
    got, k_got, v_got, ln = _run_fused(sv, hid, W, tok, None, kc, vc, kb, vb, t)
    assert_same(got, exp, "fused chain acceptance")
    assert np.array_equal(k_got, k_ref) and np.array_equal(v_got, v_ref)
    assert np.array_equal(ln, ln_ref)
    assert sv.get_device_error() == 0


def test_fused_chain_ties_across_slab_edges(sv):
    """Each row's maximum is a pair of equal columns straddling a slab edge
    (127 and 128, 255 and 256, ...): the lower column is the token."""
    B, R, H, V = 4, 5, 128, 8192
    rng = np.random.default_rng(3)
    hid = rng.integers(-2, 3, size=(B * R, H)).astype(np.float32)
    W = (rng.integers(-8, 9, size=(H, V)) * 2.0 ** -6).astype(np.float32)
    edges = [SLAB * (r + 1) for r in range(B * R)]
    for r, e in enumerate(edges):
        # 4 * sum|hid[r]| at the pair, far above any other column of row r
        W[:, e - 1] = W[:, e] = 4.0 * np.sign(hid[r])
    hid_t, W_t = _bf16(hid), _bf16(W)
    logits = _oracle_logits(hid_t, W_t).reshape(B, R, V)
    g = logits.argmax(-1)
    assert all(int(g.reshape(-1)[r]) == e - 1 for r, e in enumerate(edges))
    tok = synth.plant_chain_drafts(g, 0.8, V, seed=9)
    exp = oracle.accept_greedy(logits, tok)
    _, keys = sv.lm_head_argmax(hid_t.cuda(), W_t.cuda(), write_logits=False)
    got = sv.accept_greedy_commit(keys, torch.from_numpy(tok).cuda(), V)
    assert_same(got, exp, "fused ties at slab edges")


@pytest.mark.parametrize("seed", [0, 1])
def test_fused_tree_vs_oracle(sv, seed):
    """64-node draft trees (65 rows per sequence: the tcgen05 LM head), path
    compaction in the commit."""
    B, H, V, L, Hkv = 2, 128, 30000, 3, 2
    par = synth.random_tree(64, 8, 3, 50 + seed)
    R = len(par)
    parent = np.tile(par, (B, 1)).astype(np.int32)
    hid, W = _exact_lm(B * R, H, V, seed=77 + seed)
    logits = _oracle_logits(hid, W).reshape(B, R, V)
    g = logits.argmax(-1)
    tok = np.stack([synth.plant_tree_drafts(g[b:b + 1], par[None], 0.8, V, seed + b)[0] for b in range(B)])
    T_cap = 200
    t = np.array([T_cap - 9, 17], np.int32)[:B]
    kc, vc, kb, vb = _caches(L, B, Hkv, T_cap, R, seed=seed)
    exp = oracle.accept_greedy(logits, tok, parent)
    k_ref, v_ref, ln_ref = oracle.kv_commit(kc, vc, kb, vb, exp[2], exp[0], t)
    got, k_got, v_got, ln = _run_fused(sv, hid, W, tok, parent, kc, vc, kb, vb, t)
    assert_same(got, exp, "fused tree acceptance")
    assert np.array_equal(k_got, k_ref) and np.array_equal(v_got, v_ref)
    assert np.array_equal(ln, ln_ref)


def test_fused_acceptance_only_matches_accept_greedy(sv):
    B, R, H, V = 8, 9, 128, 20000
    hid, W = _exact_lm(B * R, H, V, seed=5)
    lg, keys = sv.lm_head_argmax(hid.cuda(), W.cuda())
    g = _oracle_logits(hid, W).reshape(B, R, V).argmax(-1)
    tok = torch.from_numpy(synth.plant_chain_drafts(g, 0.7, V, seed=2)).cuda()
    a = sv.accept_greedy(lg.reshape(B, R, V), tok)
    b = sv.accept_greedy_commit(keys, tok, V)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_fused_commit_overflow_leaves_cache(sv):
    """A sequence whose commit would pass T_cap keeps its cache and length
    (SV_DEVERR_LENGTH) but still gets its acceptance outputs."""
    B, R, H, V, L, Hkv, T_cap = 2, 5, 128, 4000, 2, 2, 64
    hid, W = _exact_lm(B * R, H, V, seed=12)
    logits = _oracle_logits(hid, W).reshape(B, R, V)
    tok = synth.plant_chain_drafts(logits.argmax(-1), 1.0, V, seed=1)   # everything accepted: 5 rows
    t = np.array([T_cap - 3, 10], np.int32)
    kc, vc, kb, vb = _caches(L, B, Hkv, T_cap, R, seed=4)
    exp = oracle.accept_greedy(logits, tok)
    got, k_got, v_got, ln = _run_fused(sv, hid, W, tok, None, kc, vc, kb, vb, t)
    assert_same(got, exp, "fused overflow acceptance")
    assert sv.get_device_error() & 0x4
    assert ln[0] == t[0] and np.array_equal(k_got[:, 0], kc[:, 0]) and np.array_equal(v_got[:, 0], vc[:, 0])
    k_ref, v_ref, ln_ref = oracle.kv_commit(kc[:, 1:], vc[:, 1:], kb[:, 1:], vb[:, 1:], exp[2][1:], exp[0][1:], t[1:])
    assert ln[1] == ln_ref[0] and np.array_equal(k_got[:, 1:], k_ref) and np.array_equal(v_got[:, 1:], v_ref)


def test_fused_nan_and_bad_token_flagged(sv):
    B, R, H, V = 1, 3, 64, 1000
    hid, W = _exact_lm(B * R, H, V, seed=8)
    hid[1, 3] = float("nan")
    tok = torch.tensor([[0, V + 3, 1]], dtype=torch.int32).cuda()
    _, keys = sv.lm_head_argmax(hid.cuda(), W.cuda(), write_logits=False)
    assert sv.get_device_error() & 0x1
    n_acc, _, _ = sv.accept_greedy_commit(keys, tok, V)
    assert sv.get_device_error() & 0x2
    assert int(n_acc[0]) == 0


def _paged_case(L, B, Hkv, M, R, seed):
    rng = np.random.default_rng(seed)
    P = B * M + 3
    kp = rng.integers(0, 65535, size=(L, P, Hkv, 64, 128), dtype=np.uint16)
    vp = rng.integers(0, 65535, size=(L, P, Hkv, 64, 128), dtype=np.uint16)
    table = rng.permutation(P)[:B * M].reshape(B, M).astype(np.int32)
    kb = rng.integers(0, 65535, size=(L, B, Hkv, R, 128), dtype=np.uint16)
    vb = rng.integers(0, 65535, size=(L, B, Hkv, R, 128), dtype=np.uint16)
    return kp, vp, table, kb, vb


@pytest.mark.parametrize("tree", [False, True])
def test_fused_paged_vs_oracle(sv, tree):
    """Acceptance from the argmax keys and the commit into paged pools in one
    launch: the oracle's acceptance, and its commit on the contiguous cache the
    page table stands for, scattered back."""
    B, H, V, L, Hkv, M = 3, 128, 20000, 2, 2, 4
    par = synth.random_tree(64, 8, 3, 61) if tree else None
    R = len(par) if tree else 5
    parent = np.tile(par, (B, 1)).astype(np.int32) if tree else None
    hid, W = _exact_lm(B * R, H, V, seed=90 + R)
    logits = _oracle_logits(hid, W).reshape(B, R, V)
    g = logits.argmax(-1)
    if tree:
        tok = np.stack([synth.plant_tree_drafts(g[b:b + 1], par[None], 0.8, V, 7 + b)[0] for b in range(B)])
    else:
        tok = synth.plant_chain_drafts(g, 0.8, V, seed=3)
    kp, vp, table, kb, vb = _paged_case(L, B, Hkv, M, R, seed=R)
    T_cap = M * 64
    t = np.array([T_cap - 9, 64 - 2, 100], np.int32)   # the last page, a page edge, the middle
    exp = oracle.accept_greedy(logits, tok, parent)
    kc_ref, vc_ref, ln_ref = oracle.kv_commit(oracle.gather_pages(kp, table), oracle.gather_pages(vp, table), kb, vb,
                                              exp[2], exp[0], t)
    kpt, vpt = _t(kp), _t(vp)
    ln = torch.from_numpy(t.copy()).cuda()
    _, keys = sv.lm_head_argmax(hid.cuda(), W.cuda(), write_logits=False)
    got = sv.accept_greedy_commit_paged(keys, torch.from_numpy(tok).cuda(), V, kpt, vpt, torch.from_numpy(table).cuda(),
                                        _t(kb), _t(vb), ln, parent=None if parent is None else
                                        torch.from_numpy(parent).cuda())
    assert_same(got, exp, "fused paged acceptance")
    assert np.array_equal(bits(kpt), oracle.scatter_pages(kp, table, kc_ref))
    assert np.array_equal(bits(vpt), oracle.scatter_pages(vp, table, vc_ref))
    assert np.array_equal(ln.cpu().numpy(), ln_ref)
    assert sv.get_device_error() == 0


def test_fused_paged_bad_page_flagged(sv):
    B, H, V, L, Hkv, M, R = 2, 128, 4000, 2, 2, 2, 5
    hid, W = _exact_lm(B * R, H, V, seed=31)
    logits = _oracle_logits(hid, W).reshape(B, R, V)
    tok = synth.plant_chain_drafts(logits.argmax(-1), 1.0, V, seed=2)   # all accepted: 5 rows each
    kp, vp, table, kb, vb = _paged_case(L, B, Hkv, M, R, seed=8)
    table[0, 1] = 10 ** 6                     # sequence 0's rows 62.. would land outside the pool
    t = np.array([62, 10], np.int32)
    kpt, vpt = _t(kp), _t(vp)
    ln = torch.from_numpy(t.copy()).cuda()
    _, keys = sv.lm_head_argmax(hid.cuda(), W.cuda(), write_logits=False)
    got = sv.accept_greedy_commit_paged(keys, torch.from_numpy(tok).cuda(), V, kpt, vpt, torch.from_numpy(table).cuda(),
                                        _t(kb), _t(vb), ln)
    assert_same(got, oracle.accept_greedy(logits, tok), "fused paged acceptance, bad page")
    assert sv.get_device_error() & 0x80
    k_got = bits(kpt)
    assert int(ln[0]) == 62 and np.array_equal(k_got[:, table[0, 0]], kp[:, table[0, 0]])
    assert int(ln[1]) == 15 and np.array_equal(k_got[:, table[1, 0], :, 10:15], kb[:, 1, :, 0:5])
