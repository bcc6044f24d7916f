"""GPU parity of sv_accept_greedy and sv_accept_sample against the oracle.

Integer outputs (n_acc, out_tok, path) must be bit-exact, given identical
logits, q and uniforms.  Inputs are seeded synthetic tensors from `synth`;
no expected value comes from the GPU.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_sv_gb300 import synth

from _helpers import assert_same

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_sv_gb300 import binding
    return binding


def _greedy_inputs(B, R, V, seed, rate=0.6, ties=False):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((B, R, V)).astype(np.float32)
    if ties:   # quantised logits: many exact ties
        logits = np.round(logits * 2).astype(np.float32)
    g = np.stack([[oracle.accept_greedy(logits[b:b + 1, j:j + 1], np.zeros((1, 1), np.int32))[1][0]
                   for j in range(R)] for b in range(B)])
    tok = synth.plant_chain_drafts(g, rate, V, seed + 1)
    return logits, tok


@pytest.mark.parametrize("B,R,V", [(1, 5, 151936), (3, 9, 152064), (16, 9, 4000), (7, 1, 1000), (2, 3, 5),
                                   (64, 9, 8192)])
def test_greedy_chain(sv, B, R, V):
    logits, tok = _greedy_inputs(B, R, V, seed=B * 1000 + R)
    got = sv.accept_greedy(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda())
    assert_same(got, oracle.accept_greedy(logits, tok), "greedy")
    assert sv.get_device_error() == 0


def test_greedy_ties_lowest_index(sv):
    logits, tok = _greedy_inputs(8, 6, 3000, seed=5, ties=True)
    got = sv.accept_greedy(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda())
    assert_same(got, oracle.accept_greedy(logits, tok), "greedy ties")


def test_greedy_golden_alignment(sv):
    g = json.load(open(os.path.join(GOLDEN, "alignment.json")))
    for case in g["cases"]:
        logits = np.array(case["logits"], np.float32)[None]
        tok = np.array(case["tok"], np.int32)[None]
        n_acc, out_tok, path = sv.accept_greedy(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda())
        assert int(n_acc[0]) == case["n_acc"], case["why"]
        assert int(out_tok[0]) == case["out_tok"], case["why"]
        assert path[0].tolist() == case["path"], case["why"]


def _tree(n_nodes, depth, seed):
    return synth.random_tree(n_nodes, depth, 3, seed)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_greedy_tree(sv, seed):
    B, V = 4, 20000
    par = _tree(64, 8, seed)
    R = len(par)
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((B, R, V)).astype(np.float32)
    g = logits.argmax(-1)
    parent = np.tile(par, (B, 1)).astype(np.int32)
    tok = np.stack([synth.plant_tree_drafts(g[b:b + 1], par[None], 0.7, V, seed + b)[0] for b in range(B)])
    got = sv.accept_greedy(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda(),
                           torch.from_numpy(parent).cuda())
    assert_same(got, oracle.accept_greedy(logits, tok, parent), "greedy tree")


def test_greedy_errors_flagged(sv):
    logits = np.zeros((1, 3, 64), np.float32)
    logits[0, 1, 5] = np.nan
    tok = np.array([[0, 99, 1]], np.int32)
    sv.accept_greedy(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda())
    word = sv.get_device_error()
    assert word & 0x1 and word & 0x2
    assert sv.get_device_error() == 0


# ----------------------------------------------------------------------------
# sampled
# ----------------------------------------------------------------------------

def _sample_case(B, k, V, Vq=None, seed=0, std=3.0, parent=None):
    return synth.sample_inputs(B, k, V, wid=100 + seed, Vq=Vq, logit_std=std, parent=parent)


@pytest.mark.parametrize("B,k,V,Vq,T", [(4, 4, 151936, None, 1.0), (8, 8, 152064, 151936, 1.0),
                                          (5, 3, 1000, None, 0.7), (3, 0, 4096, None, 1.0),
                                          (16, 8, 8192, None, 1.3), (2, 6, 4100, 4096, 0.5)])
def test_sample_chain_philox(sv, B, k, V, Vq, T):
    si = _sample_case(B, k, V, Vq, seed=B + k)
    for step in (0, 1, 2 ** 40 + 3):
        got = sv.accept_sample(si.logits.cuda(), si.q.cuda(), si.tok.cuda(), temperature=T, seed=0xDEADBEEF,
                               step=step)
        exp = oracle.accept_sample(si.logits.numpy(), si.q.numpy(), si.tok.numpy(), temperature=T,
                                   seed=0xDEADBEEF, step=step)
        assert_same(got, exp, f"sample chain step {step}")
    assert sv.get_device_error() == 0


def test_sample_chain_injected_uniforms(sv):
    B, k, V = 32, 8, 20000
    si = _sample_case(B, k, V, seed=3, std=1.0)
    rng = np.random.default_rng(4)
    for trial in range(3):
        uni = (rng.integers(0, 2 ** 24, size=(B, k + 1, 2)) * 2.0 ** -24).astype(np.float32)
        got = sv.accept_sample(si.logits.cuda(), si.q.cuda(), si.tok.cuda(), uniforms=torch.from_numpy(uni).cuda())
        exp = oracle.accept_sample(si.logits.numpy(), si.q.numpy(), si.tok.numpy(), uniforms=uni)
        assert_same(got, exp, "sample chain uniforms")


@pytest.mark.parametrize("B,k,V,T", [(48, 8, 4100, 0.7), (40, 7, 151936, 1.0), (33, 8, 20000, 1.3),
                                     (20, 8, 4096, 1.0), (24, 8, 1000, 0.9)])
def test_sample_many_rows_pipelined(sv, B, k, V, T):
    """Enough rows that the statistics CTA pairs take several rows each (the
    next row's maximum is read in the loop over the current row's sums): a
    ragged last chunk, temperatures other than 1, row counts that leave some
    pairs a row short, and one-block rows (V <= 4096: the pair's second CTA
    holds no chunk)."""
    si = _sample_case(B, k, V, seed=B + k, std=2.0)
    got = sv.accept_sample(si.logits.cuda(), si.q.cuda(), si.tok.cuda(), temperature=T, seed=77, step=3)
    exp = oracle.accept_sample(si.logits.numpy(), si.q.numpy(), si.tok.numpy(), temperature=T, seed=77, step=3)
    assert_same(got, exp, "sample many rows")
    assert sv.get_device_error() == 0


@pytest.mark.parametrize("T", [1.0, 0.8])
def test_sample_many_rows_wide_and_narrow(sv, T):
    """Rows whose z - M all lie above -86.5 (every exp(z - M) a normal number)
    and rows spanning far more, interleaved over the statistics CTAs: both
    forms of the exponential must give the oracle's bits."""
    B, k, V = 40, 8, 20000
    rng = np.random.default_rng(17)
    logits = rng.standard_normal((B, k + 1, V)).astype(np.float32) * 2
    wide = (np.arange(B * (k + 1)).reshape(B, k + 1) % 3) == 0
    logits[wide] *= 25                     # std 50: spans a few hundred
    logits[1, 2, :5] = -90.0               # just past the normal range, one row
    logits[2, 3, 7] = -80.0                # inside it
    lg = torch.from_numpy(logits)
    si = synth.sample_inputs(B, k, V, wid=130, logits=lg, logit_std=2.0)
    got = sv.accept_sample(lg.cuda(), si.q.cuda(), si.tok.cuda(), temperature=T, seed=5, step=1)
    exp = oracle.accept_sample(logits, si.q.numpy(), si.tok.numpy(), temperature=T, seed=5, step=1)
    assert_same(got, exp, "sample wide and narrow rows")
    assert sv.get_device_error() == 0


def test_sample_many_rows_nonfinite_flagged(sv):
    # a non-finite logit in a row whose maximum is taken ahead, under the
    # previous row's sums (rows past the first wave of CTAs)
    B, k, V = 40, 8, 4096
    si = _sample_case(B, k, V, seed=61)
    for bad in (float("nan"), float("inf")):
        logits = si.logits.clone()
        logits[35, 4, 1000] = bad   # row 35 * 9 + 4 = 319
        sv.accept_sample(logits.cuda(), si.q.cuda(), si.tok.cuda(), seed=1)
        assert sv.get_device_error() & 0x1


def test_sample_full_size_b64_k8(sv):
    """The sampled-acceptance workload at full size: 64 sequences, k = 8,
    vocab 151936, T = 1, target logits ~ N(0, 3^2)."""
    si = synth.sample_inputs(64, 8, 151936, wid=2)
    got = sv.accept_sample(si.logits.cuda(), si.q.cuda(), si.tok.cuda(), seed=2024, step=7)
    exp = oracle.accept_sample(si.logits.numpy(), si.q.numpy(), si.tok.numpy(), seed=2024, step=7)
    assert_same(got, exp, "sample b64")
    n_acc = exp[0]
    assert 0 < n_acc.mean() < 8   # both rejections and acceptances occur


@pytest.mark.parametrize("seed", [0, 1])
def test_sample_tree(sv, seed):
    V = 30000
    par = _tree(64, 8, seed)
    si = _sample_case(3, len(par) - 1, V, seed=10 + seed, std=1.5, parent=par)
    for step in (0, 5):
        got = sv.accept_sample(si.logits.cuda(), si.q.cuda(), si.tok.cuda(), si.parent.cuda(), seed=99, step=step)
        exp = oracle.accept_sample(si.logits.numpy(), si.q.numpy(), si.tok.numpy(), si.parent.numpy(), seed=99,
                                   step=step)
        assert_same(got, exp, "sample tree")


def test_sample_tree_with_rejected_siblings(sv):
    # q far from p so that siblings are rejected and residuals chain
    V = 8192
    par = np.array([-1, 0, 0, 0, 1, 1, 4, 4, 4], np.int32)
    B = 24
    rng = np.random.default_rng(7)
    logits = torch.from_numpy((rng.standard_normal((B, len(par), V)) * 2).astype(np.float32))
    si = synth.sample_inputs(B, len(par) - 1, V, wid=120, parent=par,
                             logits=logits, logit_std=2.0)
    q = torch.softmax(torch.from_numpy(rng.standard_normal((B, len(par), V)).astype(np.float32) * 2), -1)
    got = sv.accept_sample(logits.cuda(), q.contiguous().cuda(), si.tok.cuda(), si.parent.cuda(), seed=1, step=2)
    exp = oracle.accept_sample(logits.numpy(), q.numpy(), si.tok.numpy(), si.parent.numpy(), seed=1, step=2)
    assert_same(got, exp, "sample tree siblings")


# Draft trees of the token-tree workload (64 nodes, depth 8, up to 3 children)
# at the 7B vocabulary.  Above 32768 columns each CTA of the walking cluster
# holds several 4096-column blocks, the layout the full vocabulary runs in.
V_7B, VQ_DRAFT = 152064, 151936


def _tree_children(par):
    kids = [[] for _ in par]
    for c in range(1, len(par)):
        kids[int(par[c])].append(c)
    return kids


@pytest.mark.parametrize("Vq", [V_7B, VQ_DRAFT])
@pytest.mark.parametrize("seed", [0, 1])
def test_sample_tree_full_vocab_philox(sv, Vq, seed):
    par = _tree(64, 8, 40 + seed)
    si = _sample_case(3, len(par) - 1, V_7B, Vq=Vq, seed=60 + seed, std=1.5, parent=par)
    for step in (0, 9):
        got = sv.accept_sample(si.logits.cuda(), si.q.cuda(), si.tok.cuda(), si.parent.cuda(), seed=4242, step=step)
        exp = oracle.accept_sample(si.logits.numpy(), si.q.numpy(), si.tok.numpy(), si.parent.numpy(), seed=4242,
                                   step=step)
        assert_same(got, exp, f"sample tree V={V_7B} Vq={Vq} step {step}")
    assert sv.get_device_error() == 0


@pytest.mark.parametrize("T,B", [(0.7, 2), (1.3, 6)])
def test_sample_tree_full_vocab_temperature(sv, T, B):
    """The 64-node tree at the 7B vocabulary with a temperature other than 1:
    every pass divides the logits by T before the row's maximum, exponential
    and divisions by Z and S; at B = 2 the walk takes 16-CTA clusters, at
    B = 6 8-CTA ones."""
    par = _tree(64, 8, 52)
    si = _sample_case(B, len(par) - 1, V_7B, Vq=VQ_DRAFT, seed=70 + B, std=1.5, parent=par)
    got = sv.accept_sample(si.logits.cuda(), si.q.cuda(), si.tok.cuda(), si.parent.cuda(), temperature=T,
                           seed=515, step=7)
    exp = oracle.accept_sample(si.logits.numpy(), si.q.numpy(), si.tok.numpy(), si.parent.numpy(), temperature=T,
                               seed=515, step=7)
    assert_same(got, exp, f"sample tree T={T}")
    assert sv.get_device_error() == 0


@pytest.mark.parametrize("Vq", [V_7B, VQ_DRAFT])
def test_sample_tree_full_vocab_rejected_siblings(sv, Vq):
    """q far from p (an independent softmax): residual chains of two and
    three siblings at the full vocabulary.  Trial 0: the first children of
    every node carry the draft's most likely tokens (q well above p) and
    uniforms just below 1, so they are rejected, and the last child carries
    the target's most likely token with uniform 0, so it is accepted against
    the residual its siblings left.  Trial 1: every child carries one of the
    draft's top tokens and is rejected, so each walk ends in a resample from
    the residual of all its siblings.  Trial 2: random tokens and uniforms."""
    par = _tree(64, 8, 44)
    R, B = len(par), 4
    rng = np.random.default_rng(21)
    logits = torch.from_numpy((rng.standard_normal((B, R, V_7B)) * 2).astype(np.float32))
    q = torch.softmax(torch.from_numpy(rng.standard_normal((B, R, Vq)).astype(np.float32) * 2), -1).contiguous()
    parent = torch.from_numpy(np.tile(par, (B, 1)).astype(np.int32))
    kids = _tree_children(par)
    assert len(kids[0]) == 3
    best = logits[:, :, :Vq].argmax(-1).numpy()
    qtop = torch.topk(q, 3, dim=-1).indices.numpy()
    reject = 1.0 - 2.0 ** -24
    for trial in range(3):
        tok = rng.integers(0, Vq, size=(B, R)).astype(np.int32)
        uni = (rng.integers(0, 2 ** 24, size=(B, R, 2)) * 2.0 ** -24).astype(np.float32)
        if trial < 2:
            for u, ch in enumerate(kids):
                for i, c in enumerate(ch):
                    last = i == len(ch) - 1
                    tok[:, c] = best[:, u] if (trial == 0 and last) else qtop[:, u, i]
                    uni[:, c, 0] = 0.0 if (trial == 0 and last) else reject
        got = sv.accept_sample(logits.cuda(), q.cuda(), torch.from_numpy(tok).cuda(), parent.cuda(),
                               uniforms=torch.from_numpy(uni).cuda())
        exp = oracle.accept_sample(logits.numpy(), q.numpy(), tok, parent.numpy(), uniforms=uni)
        assert_same(got, exp, f"sample tree siblings V={V_7B} Vq={Vq} trial {trial}")
        if trial == 0:   # the root's third child was taken after two rejections
            assert all(int(exp[2][b, 1]) == kids[0][-1] for b in range(B))
        if trial == 1:   # all three of the root's children were rejected
            assert all(int(exp[0][b]) == 0 for b in range(B))
    assert sv.get_device_error() == 0


def test_sample_one_hot_equals_greedy(sv):
    B, R, V = 40, 6, 4096
    rng = np.random.default_rng(9)
    g = rng.integers(0, V, size=(B, R))
    logits = np.zeros((B, R, V), np.float32)
    np.put_along_axis(logits, g[..., None], 200.0, axis=-1)
    tok = rng.integers(0, V, size=(B, R)).astype(np.int32)
    plant = rng.random((B, R)) < 0.7
    tok[:, 1:] = np.where(plant[:, 1:], g[:, :-1], tok[:, 1:])
    q = np.zeros((B, R - 1, V), np.float32)
    np.put_along_axis(q, tok[:, 1:, None].astype(np.int64), 1.0, axis=-1)
    gs = sv.accept_greedy(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda())
    ss = sv.accept_sample(torch.from_numpy(logits).cuda(), torch.from_numpy(q).cuda(), torch.from_numpy(tok).cuda(),
                          seed=3)
    for a, b in zip(gs, ss):
        assert torch.equal(a, b)


def test_sample_errors_flagged(sv):
    B, k, V = 2, 3, 1000
    si = _sample_case(B, k, V, seed=50)
    tok = si.tok.clone()
    tok[0, 1] = V + 5
    logits = si.logits.clone()
    logits[1, 2, 17] = float("inf")
    sv.accept_sample(logits.cuda(), si.q.cuda(), tok.cuda(), seed=1)
    word = sv.get_device_error()
    assert word & 0x2 and word & 0x1


# ----------------------------------------------------------------------------
# relaxed (lossy Delta-logit) acceptance
# ----------------------------------------------------------------------------

def _relaxed_inputs(B, R, V, seed, quantise=False):
    """Drafts among the verifying row's three best tokens and random ids, so
    gaps fall on both sides of the thresholds."""
    rng = np.random.default_rng(seed)
    logits = (rng.standard_normal((B, R, V)) * 2).astype(np.float32)
    if quantise:   # many exact ties, gaps in steps of 0.5
        logits = np.round(logits * 2).astype(np.float32) / 2
    top3 = np.argsort(-logits, axis=-1, kind="stable")[..., :3]
    pick = rng.integers(0, 4, size=(B, R))
    rnd = rng.integers(0, V, size=(B, R))
    cand = np.where(pick < 3, np.take_along_axis(top3, np.minimum(pick, 2)[..., None], -1)[..., 0], rnd)
    tok = rng.integers(0, V, size=(B, R)).astype(np.int32)
    tok[:, 1:] = cand[:, :-1]
    return logits, tok


@pytest.mark.parametrize("B,R,V", [(1, 5, 151936), (16, 9, 152064), (7, 3, 1000), (64, 9, 8192)])
@pytest.mark.parametrize("delta", [0.0, 0.25, 1.0, 4.0, float("inf")])
def test_relaxed_chain(sv, B, R, V, delta):
    logits, tok = _relaxed_inputs(B, R, V, seed=B * 100 + R)
    got = sv.accept_greedy_relaxed(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda(), delta=delta)
    assert_same(got, oracle.accept_greedy_relaxed(logits, tok, delta=delta), f"relaxed chain delta {delta}")
    assert sv.get_device_error() == 0


@pytest.mark.parametrize("delta", [0.0, 0.5, 1.5])
def test_relaxed_ties_and_tree(sv, delta):
    B, V = 12, 3000
    par = _tree(40, 6, 3)
    R = len(par)
    logits, tok = _relaxed_inputs(B, R, V, seed=77, quantise=True)
    parent = np.tile(par, (B, 1)).astype(np.int32)
    for p in (None, parent):
        pt = None if p is None else torch.from_numpy(p).cuda()
        got = sv.accept_greedy_relaxed(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda(), pt, delta=delta)
        assert_same(got, oracle.accept_greedy_relaxed(logits, tok, p, delta=delta), f"relaxed tree={p is not None}")


def test_relaxed_zero_delta_equals_greedy_on_gpu(sv):
    logits, tok = _greedy_inputs(8, 9, 20000, seed=5)
    a = sv.accept_greedy(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda())
    b = sv.accept_greedy_relaxed(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda(), delta=0.0)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_relaxed_bad_token_flagged(sv):
    logits, tok = _relaxed_inputs(2, 4, 500, seed=9)
    tok[1, 2] = 600
    sv.accept_greedy_relaxed(torch.from_numpy(logits).cuda(), torch.from_numpy(tok).cuda(), delta=1.0)
    assert sv.get_device_error() & 0x2
