"""GPU parity of sv_verify_attn against the oracle (double precision):
max|err| <= 1e-2 max|ref| per call, over chain and tree masks, ragged and
empty contexts, several key tiles and splits, and full-size layers of the
Qwen2.5-1.5B / 7B workloads."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_sv_gb300 import synth

from _helpers import bits, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_sv_gb300 import binding
    return binding


def _run(sv, B, R, Hq, Hkv, T_cap, lengths, parent=None, seed=0, scale=None):
    D = 128
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    q, kc, vc, kb, vb = mk(B, R, Hq, D), mk(B, Hkv, T_cap, D), mk(B, Hkv, T_cap, D), mk(B, Hkv, R, D), mk(B, Hkv, R, D)
    ln = torch.tensor(lengths, dtype=torch.int32)
    par_t = None if parent is None else torch.from_numpy(np.ascontiguousarray(parent, np.int32))
    out = sv.verify_attn(q.cuda(), kc.cuda(), vc.cuda(), ln.cuda(), kb.cuda(), vb.cuda(),
                         None if par_t is None else par_t.cuda(), scale=scale)
    ref = oracle.verify_attn(bits(q), bits(kc), bits(vc), ln.numpy(), bits(kb), bits(vb),
                             None if par_t is None else par_t.numpy(), scale)
    return out.float().cpu().numpy(), ref


@pytest.mark.parametrize("B,R,Hq,Hkv,T_cap,lengths", [
    (1, 5, 12, 2, 2112, [2048]),                 # 1.5B layout, t = 2048
    (2, 5, 12, 2, 320, [0, 1]),                  # empty and single-key contexts
    (3, 9, 28, 4, 256, [63, 64, 65]),            # 7B layout, tile edges
    (2, 1, 8, 8, 200, [150, 7]),                 # R = 1, MHA
    (4, 9, 28, 4, 1100, [1000, 513, 1024, 77]),  # ragged batch, multiple tiles and splits
    (1, 17, 16, 2, 700, [600]),                  # 136 rows: 3 row tiles
    (2, 3, 4, 1, 130, [130, 129]),               # full cache
    (8, 17, 16, 4, 700, [600, 1, 64, 65, 300, 0, 511, 700]),   # 68 rows x 32 units: 128-row tiles
])
def test_attn_chain(sv, B, R, Hq, Hkv, T_cap, lengths):
    got, ref = _run(sv, B, R, Hq, Hkv, T_cap, lengths, seed=B * 31 + R)
    ok, err, bound = within_tol(got, ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0


@pytest.mark.parametrize("R,Hq,Hkv,lengths,tree", [
    (5, 12, 2, [2048 + 37, 100, 1], False),     # half tiles, partial last tiles
    (17, 16, 2, [600, 65], False),              # full tiles
    (65, 28, 4, [513, 300], True),              # tree, full tiles, two block tiles
])
def test_attn_cache_rows_past_len_ignored(sv, R, Hq, Hkv, lengths, tree):
    """Cache positions >= len hold NaN (K) and +inf (V) bit patterns: the
    output must not see them (P is 0 there, and 0 * inf must not reach O)."""
    B, D, T_cap = len(lengths), 128, 2304
    g = torch.Generator().manual_seed(404 + R)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    q, kc, vc, kb, vb = mk(B, R, Hq, D), mk(B, Hkv, T_cap, D), mk(B, Hkv, T_cap, D), mk(B, Hkv, R, D), mk(B, Hkv, R, D)
    kcb, vcb = kc.view(torch.int16), vc.view(torch.int16)
    for bi, t in enumerate(lengths):
        kcb[bi, :, t:] = 0x7FC0        # NaN
        vcb[bi, :, t:] = 0x7F80        # +inf
    ln = torch.tensor(lengths, dtype=torch.int32)
    par = None
    if tree:
        par = np.tile(synth.random_tree(R - 1, 8, 3, 5), (B, 1)).astype(np.int32)
    out = sv.verify_attn(q.cuda(), kc.cuda(), vc.cuda(), ln.cuda(), kb.cuda(), vb.cuda(),
                         None if par is None else torch.from_numpy(par).cuda())
    got = out.float().cpu().numpy()
    ref = oracle.verify_attn(bits(q), bits(kc), bits(vc), ln.numpy(), bits(kb), bits(vb), par)
    assert np.isfinite(got).all()
    ok, err, bound = within_tol(got, ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0


@pytest.mark.parametrize("B,R,Hq,Hkv,T_cap,t", [(1, 5, 12, 2, 4160, 4096), (16, 9, 28, 4, 1152, 1000),
                                                 (2, 65, 28, 4, 704, 600)])
def test_attn_cache_ready_same_result(sv, B, R, Hq, Hkv, T_cap, t):
    """Layers of one round back to back on a stream, the later ones launched
    with SV_ATTN_CACHE_READY (length and cache read before the preceding
    kernel completes): every layer's output equals the flag-free launch,
    bit for bit."""
    D, L = 128, 4
    g = torch.Generator().manual_seed(B * 7 + R)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16).cuda()
    q, kc, vc = mk(L, B, R, Hq, D), mk(L, B, Hkv, T_cap, D), mk(L, B, Hkv, T_cap, D)
    kb, vb = mk(L, B, Hkv, R, D), mk(L, B, Hkv, R, D)
    ln = torch.full((B,), t, dtype=torch.int32).cuda()
    par = None
    if R > 9:
        par = torch.from_numpy(np.tile(synth.random_tree(R - 1, 8, 3, 1), (B, 1)).astype(np.int32)).cuda()
    ws = torch.zeros(max(sv.verify_attn_workspace(B, R, Hq, Hkv, D, T_cap), 16), dtype=torch.uint8, device="cuda")
    ref = [sv.verify_attn(q[l], kc[l], vc[l], ln, kb[l], vb[l], par, ws=ws) for l in range(L)]
    torch.cuda.synchronize()
    out = torch.empty(L, B, R, Hq, D, dtype=torch.bfloat16, device="cuda")
    for l in range(L):
        sv.verify_attn(q[l], kc[l], vc[l], ln, kb[l], vb[l], par, out=out[l], ws=ws, cache_ready=l > 0)
    torch.cuda.synchronize()
    for l in range(L):
        assert torch.equal(out[l], ref[l]), l
    assert sv.get_device_error() == 0


def test_attn_custom_scale(sv):
    got, ref = _run(sv, 2, 5, 12, 2, 400, [300, 211], seed=3, scale=0.21)
    ok, err, bound = within_tol(got, ref)
    assert ok, (err, bound)


@pytest.mark.parametrize("seed", [0, 1])
def test_attn_tree_65_nodes(sv, seed):
    par = synth.random_tree(64, 8, 3, seed)
    B = 2
    parent = np.tile(par, (B, 1))
    got, ref = _run(sv, B, 65, 28, 4, 600, [513, 300], parent=parent, seed=seed + 50)
    ok, err, bound = within_tol(got, ref)
    assert ok, (err, bound)


@pytest.mark.parametrize("B,R,Hq,Hkv,lengths,tree", [
    (8, 17, 16, 4, [600, 1, 64, 65, 300, 0, 511, 700], False),   # 68 rows: quadrants 0-2 live, 4 rows in 2
    (8, 10, 32, 4, [600, 513, 64, 0, 700, 1, 65, 300], False),   # 80 rows, 8 heads per group
    (8, 24, 16, 4, [600, 300, 0, 700, 1, 64, 65, 511], False),   # 96 rows: quadrant 3 dead
    (8, 30, 16, 4, [700, 600, 1, 0, 65, 64, 300, 513], False),   # 120 rows: padding inside quadrant 3
    (8, 33, 16, 4, [600, 0, 700, 64, 1, 65, 511, 300], False),   # 132 rows: a full tile and a 4-row tile
    (4, 33, 16, 4, [600, 0, 700, 65], True),                     # the same under a tree mask
    (2, 65, 28, 4, [700, 513], True),                            # the draft tree at batch 2 (4-CTA clusters)
])
def test_attn_full_tile_row_counts(sv, B, R, Hq, Hkv, lengths, tree):
    """128-row tiles (two key tiles per step, split K/V barriers) with every
    count of live TMEM quadrants and padding rows inside a live quadrant,
    chains and trees, against the oracle (the plan takes full tiles for these
    shapes, in clusters of 4 or 2)."""
    parent = None
    if tree:
        parent = np.tile(synth.random_tree(R - 1, 8, 3, R), (B, 1))
    got, ref = _run(sv, B, R, Hq, Hkv, 704, lengths, parent=parent, seed=B * 13 + R)
    ok, err, bound = within_tol(got, ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0


@pytest.mark.parametrize("B,R,Hq,Hkv,T_cap,lengths,tree", [
    (1, 17, 16, 2, 704, [600], False),                 # half tiles, 12-CTA clusters
    (1, 33, 16, 4, 704, [650], False),                 # full tiles, 12-CTA clusters
    (3, 33, 16, 4, 1408, [1300, 1, 700], False),       # full tiles, 5-CTA clusters
    (1, 65, 28, 4, 1408, [1300], True),                # the draft tree, full tiles, 6-CTA clusters
])
def test_attn_cluster_sizes(sv, B, R, Hq, Hkv, T_cap, lengths, tree):
    """Shapes whose plan picks a cluster size that is not a power of two
    (split bounds, light owners and the merge over C CTAs)."""
    parent = np.tile(synth.random_tree(R - 1, 8, 3, 7), (B, 1)) if tree else None
    got, ref = _run(sv, B, R, Hq, Hkv, T_cap, lengths, parent=parent, seed=B * 17 + R)
    ok, err, bound = within_tol(got, ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0


@pytest.mark.parametrize("seed", [3, 4])
def test_attn_tree_small_unit(sv, seed):
    """A 9-node tree with 3 query heads per KV head: 27 query rows per
    (sequence, KV head), the half-tile layout under a tree mask, with an
    empty-ish context (t = 1) in the batch."""
    par = synth.random_tree(8, 4, 3, seed)
    B = 3
    parent = np.tile(par, (B, 1))
    got, ref = _run(sv, B, 9, 12, 4, 600, [513, 1, 300], parent=parent, seed=seed + 70)
    ok, err, bound = within_tol(got, ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0


def test_attn_chain_equals_path_tree(sv):
    B, R = 2, 9
    parent = np.tile(np.arange(-1, R - 1, dtype=np.int32), (B, 1))
    a, ref = _run(sv, B, R, 28, 4, 300, [250, 100], seed=77)
    b, _ = _run(sv, B, R, 28, 4, 300, [250, 100], parent=parent, seed=77)
    assert np.array_equal(a, b)
    assert within_tol(a, ref)[0]


def test_attn_bad_length_flagged(sv):
    got, ref = _run(sv, 1, 3, 4, 1, 64, [64], seed=9)
    assert within_tol(got, ref)[0]
    D = 128
    q = torch.randn(1, 3, 4, D).to(torch.bfloat16).cuda()
    kc = torch.randn(1, 1, 64, D).to(torch.bfloat16).cuda()
    sv.verify_attn(q, kc, kc, torch.tensor([65], dtype=torch.int32).cuda(), kc[:, :, :3].contiguous(),
                   kc[:, :, :3].contiguous())
    assert sv.get_device_error() & 0x4


@pytest.mark.parametrize("wid,B,layer", [(0, 1, 0), (1, 1, 27), (3, 1, 5), (3, 16, 0)])
def test_attn_full_layer(sv, wid, B, layer):
    """A full-size layer of the 1.5B / 7B workloads, generated on the GPU; the
    oracle checks every output row of sequences 0 and B-1."""
    w = synth.workload(wid, B=B)
    ai = synth.attn_inputs(w, device="cuda", layers=layer + 1)
    L = layer
    out = sv.verify_attn(ai.q[L], ai.k_cache[L], ai.v_cache[L], ai.length, ai.k_blk[L], ai.v_blk[L])
    for b in sorted({0, B - 1}):
        ref = oracle.verify_attn(bits(ai.q[L, b:b + 1]), bits(ai.k_cache[L, b:b + 1]), bits(ai.v_cache[L, b:b + 1]),
                                 ai.length[b:b + 1].cpu().numpy(), bits(ai.k_blk[L, b:b + 1]),
                                 bits(ai.v_blk[L, b:b + 1]))
        ok, err, bound = within_tol(out[b:b + 1].float().cpu().numpy(), ref)
        assert ok, (b, err, bound)


def test_attn_full_tree_layer(sv):
    """A full-size layer of the 7B tree workload (64 draft nodes, depth 8,
    t = 8192): 455 query rows per KV head in eight half tiles, each CTA
    streaming enough key tiles for four row-owner warps per quadrant; every
    output row is checked against the oracle."""
    w = synth.workload(4)
    ai = synth.attn_inputs(w, device="cuda", layers=1)
    par = np.stack([synth.random_tree(w.R - 1, w.tree_depth, 3, synth.seed_for(w.wid, 12 + b))
                    for b in range(w.B)]).astype(np.int32)
    out = sv.verify_attn(ai.q[0], ai.k_cache[0], ai.v_cache[0], ai.length, ai.k_blk[0], ai.v_blk[0],
                         torch.from_numpy(par).cuda())
    ref = oracle.verify_attn(bits(ai.q[0]), bits(ai.k_cache[0]), bits(ai.v_cache[0]), ai.length.cpu().numpy(),
                             bits(ai.k_blk[0]), bits(ai.v_blk[0]), par)
    ok, err, bound = within_tol(out.float().cpu().numpy(), ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0


def test_attn_workspace_multi_row_tiles(sv):
    """72 query rows per KV head over a 32K context (one 128-row tile or two
    half tiles, as the plan costs them): several clusters per (KV head, row
    tile) meet in the workspace; the merged rows match the oracle and the
    tickets end at zero."""
    B, R, Hq, Hkv, T_cap = 1, 9, 8, 1, 32832
    nbytes = sv.verify_attn_workspace(B, R, Hq, Hkv, 128, T_cap)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    g = torch.Generator().manual_seed(13)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    q, kc, vc = mk(B, R, Hq, 128), mk(B, Hkv, T_cap, 128), mk(B, Hkv, T_cap, 128)
    kb, vb = mk(B, Hkv, R, 128), mk(B, Hkv, R, 128)
    ln = torch.tensor([32700], dtype=torch.int32)
    out = sv.verify_attn(q.cuda(), kc.cuda(), vc.cuda(), ln.cuda(), kb.cuda(), vb.cuda(), ws=ws)
    torch.cuda.synchronize()
    assert int(ws[:256].view(torch.int32).abs().sum()) == 0
    ref = oracle.verify_attn(bits(q), bits(kc), bits(vc), ln.numpy(), bits(kb), bits(vb))
    ok, err, bound = within_tol(out.float().cpu().numpy(), ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0


def test_attn_workspace_full_tile_tree(sv):
    """A 64-node draft tree with 7 query heads on one KV head (455 rows: four
    128-row tiles) over a 16K context: the plan splits each tile over several
    clusters of a size that is not a power of two, which meet in the workspace
    under the tree mask."""
    B, R, Hq, Hkv, T_cap = 1, 65, 7, 1, 16448
    assert sv.verify_attn_workspace(B, R, Hq, Hkv, 128, T_cap) > 0   # several clusters per tile
    par = synth.random_tree(R - 1, 8, 3, 21)[None, :]
    got, ref = _run(sv, B, R, Hq, Hkv, T_cap, [16300], parent=par, seed=29)
    ok, err, bound = within_tol(got, ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0


@pytest.mark.parametrize("B,R,Hq,Hkv,T_cap,lengths,tree", [
    (1, 65, 7, 1, 32832, [32700], True),          # a 64-node tree on one KV head: 4 tiles x ~7 clusters of 5
    (2, 33, 7, 1, 32832, [32000, 20013], False),   # 231-row chains: 2 tiles per sequence, several clusters each
])
def test_attn_workspace_exchange(sv, B, R, Hq, Hkv, T_cap, lengths, tree):
    """128-row tiles split over several clusters of at most six CTAs: each
    cluster's CTAs meet through the L2 exchange area, and the clusters'
    merged partials through the workspace tickets, in one launch."""
    assert sv.verify_attn_workspace(B, R, Hq, Hkv, 128, T_cap) > 0
    parent = np.tile(synth.random_tree(R - 1, 8, 3, 31), (B, 1)) if tree else None
    got, ref = _run(sv, B, R, Hq, Hkv, T_cap, lengths, parent=parent, seed=B * 41 + R)
    ok, err, bound = within_tol(got, ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0


def test_attn_workspace_tickets_reset(sv):
    """A batch-1, 32K-context layer splits each KV head over several clusters
    that meet in the workspace through a ticket word; every call must leave
    the tickets at zero so one workspace serves consecutive calls (same result
    as a fresh one), and the merged rows match the oracle."""
    B, R, Hq, Hkv, T_cap = 1, 5, 12, 2, 32832
    nbytes = sv.verify_attn_workspace(B, R, Hq, Hkv, 128, T_cap)
    assert nbytes > 0
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    g = torch.Generator().manual_seed(11)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16).cuda()
    kc, vc, kb, vb = mk(B, Hkv, T_cap, 128), mk(B, Hkv, T_cap, 128), mk(B, Hkv, R, 128), mk(B, Hkv, R, 128)
    ln = torch.tensor([32768], dtype=torch.int32, device="cuda")
    for it in range(3):
        q = mk(B, R, Hq, 128)
        shared = sv.verify_attn(q, kc, vc, ln, kb, vb, ws=ws)
        fresh = sv.verify_attn(q, kc, vc, ln, kb, vb)
        torch.cuda.synchronize()
        assert torch.equal(shared, fresh), it
        assert int(ws[:4 * B * Hkv].view(torch.int32).abs().sum()) == 0
    ref = oracle.verify_attn(bits(q.cpu()), bits(kc.cpu()), bits(vc.cpu()), ln.cpu().numpy(), bits(kb.cpu()),
                             bits(vb.cpu()))
    ok, err, bound = within_tol(shared.float().cpu().numpy(), ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0


# ----------------------------------------------------------------------------
# paged cache: the pool's pages in a shuffled order, a page table per
# sequence; the oracle attends over the contiguous cache the table stands for
# ----------------------------------------------------------------------------

def _paged_case(B, R, Hq, Hkv, max_pages, lengths, seed, spare=3, poison=False):
    D, PG = 128, 64
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: torch.randn(*s, generator=g).to(torch.bfloat16)
    P = B * max_pages + spare
    kp, vp = mk(P, Hkv, PG, D), mk(P, Hkv, PG, D)
    table = torch.randperm(P, generator=g)[:B * max_pages].reshape(B, max_pages).to(torch.int32)
    if poison:   # positions at or past len hold NaN (K) and +inf (V) bits
        for b, t in enumerate(lengths):
            for p in range(t, max_pages * PG):
                kp[table[b, p // PG], :, p % PG] = float("nan")
                vp[table[b, p // PG], :, p % PG] = float("inf")
    q, kb, vb = mk(B, R, Hq, D), mk(B, Hkv, R, D), mk(B, Hkv, R, D)
    return q, kp, vp, table, torch.tensor(lengths, dtype=torch.int32), kb, vb


@pytest.mark.parametrize("B,R,Hq,Hkv,max_pages,lengths,tree,poison", [
    (1, 5, 12, 2, 33, [2048], False, False),               # 1.5B layout over 33 pages
    (3, 9, 28, 4, 5, [63, 64, 300], False, True),           # tile edges, NaN/+inf past len
    (4, 9, 28, 4, 18, [1000, 513, 1024, 0], False, False),  # ragged, empty context
    (2, 65, 28, 4, 9, [513, 300], True, True),              # tree, two block tiles
])
def test_attn_paged(sv, B, R, Hq, Hkv, max_pages, lengths, tree, poison):
    q, kp, vp, table, ln, kb, vb = _paged_case(B, R, Hq, Hkv, max_pages, lengths, seed=B + R, poison=poison)
    par = None
    if tree:
        par = np.tile(synth.random_tree(R - 1, 8, 3, 4), (B, 1)).astype(np.int32)
    out = sv.verify_attn_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), ln.cuda(), kb.cuda(), vb.cuda(),
                               None if par is None else torch.from_numpy(par).cuda())
    kc = oracle.gather_pages(bits(kp), table.numpy())
    vc = oracle.gather_pages(bits(vp), table.numpy())
    ref = oracle.verify_attn(bits(q), kc, vc, ln.numpy(), bits(kb), bits(vb), par)
    ok, err, bound = within_tol(out.float().cpu().numpy(), ref)
    assert ok, (err, bound)
    assert sv.get_device_error() == 0
    # the same with the cache-ready launch flag: bit for bit
    out2 = sv.verify_attn_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), ln.cuda(), kb.cuda(), vb.cuda(),
                                None if par is None else torch.from_numpy(par).cuda(), cache_ready=True)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_attn_paged_equals_contiguous(sv):
    """A table that maps sequence b's tile j to page b * max_pages + j makes the
    pool the contiguous cache: both entry points give the same bits."""
    B, R, Hq, Hkv, M = 2, 9, 28, 4, 6
    q, kp, vp, _, ln, kb, vb = _paged_case(B, R, Hq, Hkv, M, [300, 129], seed=3, spare=0)
    table = torch.arange(B * M, dtype=torch.int32).reshape(B, M)
    paged = sv.verify_attn_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), ln.cuda(), kb.cuda(), vb.cuda())
    kc = kp.reshape(B, M, Hkv, 64, 128).transpose(1, 2).reshape(B, Hkv, M * 64, 128).contiguous()
    vc = vp.reshape(B, M, Hkv, 64, 128).transpose(1, 2).reshape(B, Hkv, M * 64, 128).contiguous()
    flat = sv.verify_attn(q.cuda(), kc.cuda(), vc.cuda(), ln.cuda(), kb.cuda(), vb.cuda())
    assert torch.equal(paged.view(torch.int16), flat.view(torch.int16))


def test_attn_paged_bad_page_flagged(sv):
    q, kp, vp, table, ln, kb, vb = _paged_case(1, 5, 12, 2, 4, [200], seed=8)
    table[0, 1] = kp.shape[0] + 5          # a page the context reaches, outside the pool
    sv.verify_attn_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), ln.cuda(), kb.cuda(), vb.cuda())
    assert sv.get_device_error() & 0x80
