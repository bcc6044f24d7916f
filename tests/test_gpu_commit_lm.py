"""GPU parity of sv_kv_commit (bit-exact cache and length) and sv_lm_head
(max|err| <= 1e-2 max|ref| against the oracle's double-precision product)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_sv_gb300 import synth

from _helpers import bits, within_tol

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_sv_gb300 import binding
    return binding


def _bf16_from_bits(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)


def test_commit_golden(sv):
    g = json.load(open(os.path.join(GOLDEN, "commit.json")))
    T_cap, R = g["T_cap"], g["R"]
    for case in g["cases"]:
        # D must be a multiple of 8: widen each slot to 8 equal lanes
        kc = np.repeat(np.array(case["cache_before"], np.uint16)[:, None], 8, 1).reshape(1, 1, 1, T_cap, 8)
        kb = np.repeat(np.array(case["block"], np.uint16)[:, None], 8, 1).reshape(1, 1, 1, R, 8)
        kct, vct = _bf16_from_bits(kc).cuda(), _bf16_from_bits(kc + 1000).cuda()
        ln = torch.tensor([case["t"]], dtype=torch.int32).cuda()
        sv.kv_commit(kct, vct, _bf16_from_bits(kb).cuda(), _bf16_from_bits(kb + 1000).cuda(),
                     torch.tensor([case["path"]], dtype=torch.int32).cuda(),
                     torch.tensor([case["n_acc"]], dtype=torch.int32).cuda(), ln)
        got = bits(kct).reshape(T_cap, 8)[:, 0]
        assert got.tolist() == case["cache_after"], case["why"]
        assert (bits(vct).reshape(T_cap, 8)[:, 0] - 1000).tolist() == case["cache_after"], case["why"]
        assert int(ln[0]) == case["len_after"], case["why"]


@pytest.mark.parametrize("L,B,Hkv,T_cap,R,tree", [(3, 5, 2, 128, 5, False), (28, 16, 4, 8320, 9, False),
                                                  (2, 4, 4, 300, 65, True), (1, 1, 2, 64, 1, False)])
def test_commit_random(sv, L, B, Hkv, T_cap, R, tree):
    D = 128
    rng = np.random.default_rng(L * 100 + B)
    shape_c = (L, B, Hkv, T_cap, D)
    kc = rng.integers(0, 65535, size=shape_c, dtype=np.uint16)
    vc = rng.integers(0, 65535, size=shape_c, dtype=np.uint16)
    kb = rng.integers(0, 65535, size=(L, B, Hkv, R, D), dtype=np.uint16)
    vb = rng.integers(0, 65535, size=(L, B, Hkv, R, D), dtype=np.uint16)
    t = rng.integers(0, T_cap - R + 1, size=B).astype(np.int32)
    t[0] = T_cap - R       # full up to the last slot when every draft is accepted
    n_acc = rng.integers(0, R, size=B).astype(np.int32)
    n_acc[0] = R - 1
    path = np.full((B, R), -1, np.int32)
    if tree:
        par = synth.random_tree(R - 1, 8, 3, 5)
        for b in range(B):
            node = int(rng.integers(0, R))
            chain = []
            while node >= 0:
                chain.append(node)
                node = int(par[node])
            chain = chain[::-1]
            n_acc[b] = len(chain) - 1
            path[b, :len(chain)] = chain
    else:
        for b in range(B):
            path[b, :n_acc[b] + 1] = np.arange(n_acc[b] + 1)
    kct, vct = _bf16_from_bits(kc).cuda(), _bf16_from_bits(vc).cuda()
    ln = torch.from_numpy(t).cuda()
    sv.kv_commit(kct, vct, _bf16_from_bits(kb).cuda(), _bf16_from_bits(vb).cuda(), torch.from_numpy(path).cuda(),
                 torch.from_numpy(n_acc).cuda(), ln)
    k_ref, v_ref, ln_ref = oracle.kv_commit(kc, vc, kb, vb, path, n_acc, t)
    assert np.array_equal(ln.cpu().numpy(), ln_ref)
    assert np.array_equal(bits(kct), k_ref)
    assert np.array_equal(bits(vct), v_ref)
    assert sv.get_device_error() == 0


def test_commit_overflow_flagged_and_untouched(sv):
    L, B, Hkv, T_cap, R, D = 1, 2, 1, 16, 4, 128
    kc = torch.randn(L, B, Hkv, T_cap, D).to(torch.bfloat16).cuda()
    before = kc.clone()
    kb = torch.randn(L, B, Hkv, R, D).to(torch.bfloat16).cuda()
    ln = torch.tensor([14, 3], dtype=torch.int32).cuda()
    path = torch.tensor([[0, 1, 2, 3], [0, 1, -1, -1]], dtype=torch.int32).cuda()
    n_acc = torch.tensor([3, 1], dtype=torch.int32).cuda()
    sv.kv_commit(kc, kc.clone(), kb, kb, path, n_acc, ln)
    assert sv.get_device_error() & 0x4
    assert ln.tolist() == [14, 5]
    assert torch.equal(kc[:, 0], before[:, 0])


# ----------------------------------------------------------------------------
# LM head
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("N,H,V", [(1, 64, 1024), (5, 1536, 4096), (9, 3584, 2048), (16, 1536, 8200),
                                   (17, 512, 1024), (65, 3584, 1536), (144, 3584, 1024), (3, 72, 136)])
def test_lm_head_small(sv, N, H, V):
    g = torch.Generator().manual_seed(N * 7 + H)
    hid = torch.randn(N, H, generator=g).to(torch.bfloat16)
    W = (torch.randn(H, V, generator=g) * 0.02).to(torch.bfloat16)
    got = sv.lm_head(hid.cuda(), W.cuda()).cpu().numpy()
    ref = oracle.lm_head(bits(hid), bits(W))
    ok, err, bound = within_tol(got, ref)
    assert ok, (err, bound)
    assert err < 1e-4 * np.max(np.abs(ref))   # fp32 accumulation is far inside the bar


@pytest.mark.parametrize("wid,B", [(0, 1), (3, 1), (3, 16)])
def test_lm_head_full_shape_sampled_columns(sv, wid, B):
    w = synth.workload(wid, B=B)
    hid, W = synth.lm_inputs(w, device="cuda")
    got = sv.lm_head(hid, W)
    cols = [(0, 512), (w.V // 2 - 256, w.V // 2 + 256), (w.V - 640, w.V)]
    hid_b, W_c = bits(hid), None
    for v0, v1 in cols:
        W_c = bits(W[:, v0:v1].contiguous())
        ref = oracle.lm_head(hid_b, W_c)
        ok, err, bound = within_tol(got[:, v0:v1].cpu().numpy(), ref)
        assert ok, (v0, err, bound)


@pytest.mark.parametrize("N,H,V", [(5, 1536, 151936), (9, 3584, 8200), (65, 3584, 4096), (144, 3584, 2048)])
def test_lm_head_weights_ready_same_result(sv, N, H, V):
    """SV_LM_WEIGHTS_READY (W loaded before the preceding kernel completes):
    launched right after another LM head on the stream, the logits equal a
    flag-free launch bit for bit, for both kernels (<= 16 rows, tcgen05)."""
    g = torch.Generator().manual_seed(N + H)
    hid = [torch.randn(N, H, generator=g).to(torch.bfloat16).cuda() for _ in range(2)]
    W = (torch.randn(H, V, generator=g) * 0.02).to(torch.bfloat16).cuda()
    ref = [sv.lm_head(h, W) for h in hid]
    torch.cuda.synchronize()
    out = [torch.empty(N, V, dtype=torch.float32, device="cuda") for _ in range(2)]
    sv.lm_head(hid[0], W, logits=out[0])
    sv.lm_head(hid[1], W, logits=out[1], weights_ready=True)
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("L,B,Hkv,max_pages,R,tree", [(3, 5, 2, 3, 5, False), (28, 4, 4, 4, 9, False),
                                                      (2, 3, 4, 5, 65, True)])
def test_commit_paged(sv, L, B, Hkv, max_pages, R, tree):
    """Paged commit equals the oracle's commit on the contiguous cache the page
    table stands for, scattered back; pages no table names are untouched."""
    D, PG = 128, 64
    rng = np.random.default_rng(L * 10 + B)
    P = B * max_pages + 4
    kp = rng.integers(0, 65535, size=(L, P, Hkv, PG, D), dtype=np.uint16)
    vp = rng.integers(0, 65535, size=(L, P, Hkv, PG, D), dtype=np.uint16)
    table = rng.permutation(P)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    kb = rng.integers(0, 65535, size=(L, B, Hkv, R, D), dtype=np.uint16)
    vb = rng.integers(0, 65535, size=(L, B, Hkv, R, D), dtype=np.uint16)
    T_cap = max_pages * PG
    t = rng.integers(0, T_cap - R + 1, size=B).astype(np.int32)
    t[0] = T_cap - R
    n_acc = rng.integers(0, R, size=B).astype(np.int32)
    path = np.full((B, R), -1, np.int32)
    for b in range(B):
        if tree:   # a strictly increasing node path, as a tree walk produces
            path[b, :n_acc[b] + 1] = np.concatenate([[0], np.sort(rng.choice(np.arange(1, R), n_acc[b], False))])
        else:
            path[b, :n_acc[b] + 1] = np.arange(n_acc[b] + 1)
    kc_ref, vc_ref, ln_ref = oracle.kv_commit(oracle.gather_pages(kp, table), oracle.gather_pages(vp, table), kb, vb,
                                              path, n_acc, t)
    kp_ref = oracle.scatter_pages(kp, table, kc_ref)
    vp_ref = oracle.scatter_pages(vp, table, vc_ref)
    kpt, vpt = _bf16_from_bits(kp).cuda(), _bf16_from_bits(vp).cuda()
    ln = torch.from_numpy(t.copy()).cuda()
    sv.kv_commit_paged(kpt, vpt, torch.from_numpy(table).cuda(), _bf16_from_bits(kb).cuda(),
                       _bf16_from_bits(vb).cuda(), torch.from_numpy(path).cuda(), torch.from_numpy(n_acc).cuda(), ln)
    assert np.array_equal(bits(kpt), kp_ref)
    assert np.array_equal(bits(vpt), vp_ref)
    assert np.array_equal(ln.cpu().numpy(), ln_ref)
    assert sv.get_device_error() == 0


def test_commit_paged_bad_page_flagged_and_untouched(sv):
    D, PG, L, B, Hkv, M, R = 128, 64, 2, 2, 2, 2, 5
    rng = np.random.default_rng(5)
    P = B * M
    kp = rng.integers(0, 65535, size=(L, P, Hkv, PG, D), dtype=np.uint16)
    table = np.arange(P, dtype=np.int32).reshape(B, M)
    table[0, 1] = P + 7                       # sequence 0's rows 62.. land on a page outside the pool
    kb = rng.integers(0, 65535, size=(L, B, Hkv, R, D), dtype=np.uint16)
    t = np.array([62, 10], np.int32)
    n_acc = np.array([3, 2], np.int32)
    path = np.array([[0, 1, 2, 3, -1], [0, 1, 2, -1, -1]], np.int32)
    kpt = _bf16_from_bits(kp).cuda()
    vpt = _bf16_from_bits(kp).cuda()
    ln = torch.from_numpy(t.copy()).cuda()
    sv.kv_commit_paged(kpt, vpt, torch.from_numpy(table).cuda(), _bf16_from_bits(kb).cuda(), _bf16_from_bits(kb).cuda(),
                       torch.from_numpy(path).cuda(), torch.from_numpy(n_acc).cuda(), ln)
    assert sv.get_device_error() & 0x80
    got = bits(kpt)
    assert np.array_equal(got[:, 0], kp[:, 0])            # sequence 0 untouched (its page 0 too)
    assert int(ln[0]) == 62 and int(ln[1]) == 13           # sequence 1 committed
    assert np.array_equal(got[:, 2, :, 10:13], kb[:, 1, :, 0:3])
