"""Pins for the oracle's greedy and sampled acceptance.

Greedy ([SpecDec-Context-Scaling guide, sec. 3 and 3.1]): hand-built golden
cases for the saved_next / rows[j-1] alignment (including the off-by-one that
"runs but is wrong"), ties, and reductions (a one-child-per-node tree is the
chain; one-hot p and q make sampling greedy).

Sampled ([wmrh.cn tutorial, sec. 2.2]; [mini-infer Phase 11, "Modified
Rejection Sampling"]; [SubSpec summary, sec. 4.2] for trees): the output
distribution of the implementation is computed EXACTLY on a 5-token vocab by
running the oracle over every one of the 2^24 values each uniform can take,
and must equal the target distribution p.  An exact-rational derivation of
the algorithm shows the identity holds with no rounding at all.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GRID = 2 ** 24
U_MAX = np.float32(1.0 - 2.0 ** -24)


# ----------------------------------------------------------------------------
# greedy
# ----------------------------------------------------------------------------


# Relaxed, lossy acceptance ([SpecDec-Context-Scaling guide, sec. 7.2], the
# Delta-logit relaxation): pinned by a hand-worked case, by its reductions to
# greedy acceptance (delta = 0 with distinct maxima) and to "accept everything"
# (delta = inf), by monotonicity in delta, and by the tie case where it and
# greedy must differ.

def test_relaxed_hand_worked_case():
    # row 0: top-1 5.0 at id 0; draft 1 has 4.5, a gap of exactly 0.5.
    # row 1: top-1 3.0 at id 2; draft 2 is id 3 with float32(2.9), gap
    #        3.0 - 2.9000000953674316 = 0.0999999046325684 (exact).
    # row 2: top-1 9 at id 3 (the bonus row).
    logits = np.array([[[5.0, 4.5, 1.0, 0.0], [0.0, 2.0, 3.0, 2.9], [1.0, 1.0, 1.0, 9.0]]], np.float32)
    tok = np.array([[0, 1, 3]], np.int32)
    cases = {
        0.4: (0, 0, [0, -1, -1]),      # gap 0.5 > 0.4: reject d_1, replacement = top-1 of row 0
        0.5: (2, 3, [0, 1, 2]),        # 0.5 <= 0.5 and 0.09999990 <= 0.5: all pass, bonus from row 2
        0.0999999: (0, 0, [0, -1, -1]),
    }
    for delta, (m, out, path) in cases.items():
        n_acc, out_tok, pth = oracle.accept_greedy_relaxed(logits, tok, delta=delta)
        assert (int(n_acc[0]), int(out_tok[0]), pth[0].tolist()) == (m, out, path), delta
    # gap of row 1 against delta just below and at it
    logits2 = logits.copy()
    logits2[0, 0, 1] = 5.0          # draft 1 is now tied with the top-1 (gap 0)
    gap1 = np.float32(3.0) - np.float32(2.9)
    n_acc, out_tok, _ = oracle.accept_greedy_relaxed(logits2, tok, delta=float(np.nextafter(gap1, np.float32(0))))
    assert (int(n_acc[0]), int(out_tok[0])) == (1, 2)   # d_1 passes at gap 0, d_2 fails: replacement id 2
    n_acc, out_tok, _ = oracle.accept_greedy_relaxed(logits2, tok, delta=float(gap1))
    assert (int(n_acc[0]), int(out_tok[0])) == (2, 3)


def test_relaxed_zero_delta_is_greedy_when_maxima_are_unique():
    rng = np.random.default_rng(31)
    B, R, V = 24, 9, 500
    logits = rng.standard_normal((B, R, V)).astype(np.float32)
    g = logits.argmax(-1)
    tok = rng.integers(0, V, size=(B, R)).astype(np.int32)
    plant = rng.random((B, R)) < 0.7
    tok[:, 1:] = np.where(plant[:, 1:], g[:, :-1], tok[:, 1:])
    for got, exp in zip(oracle.accept_greedy_relaxed(logits, tok, delta=0.0), oracle.accept_greedy(logits, tok)):
        assert np.array_equal(got, exp)
    par = np.array([-1, 0, 0, 1, 1, 2, 3, 3, 5], np.int32)
    parent = np.tile(par, (B, 1))
    for got, exp in zip(oracle.accept_greedy_relaxed(logits, tok, parent, delta=0.0),
                        oracle.accept_greedy(logits, tok, parent)):
        assert np.array_equal(got, exp)


def test_relaxed_infinite_delta_accepts_every_draft():
    rng = np.random.default_rng(32)
    B, R, V = 6, 7, 300
    logits = (rng.standard_normal((B, R, V)) * 10).astype(np.float32)
    tok = rng.integers(0, V, size=(B, R)).astype(np.int32)
    n_acc, out_tok, path = oracle.accept_greedy_relaxed(logits, tok, delta=float("inf"))
    assert (n_acc == R - 1).all()
    assert (path == np.arange(R)).all()
    assert (out_tok == logits[:, R - 1].argmax(-1)).all()     # the bonus row's top-1
    # a tree: the walk takes the first child (index order) at every node
    par = np.array([-1, 0, 0, 1, 1, 3, 2], np.int32)
    n_acc, _, path = oracle.accept_greedy_relaxed(logits, tok, np.tile(par, (B, 1)), delta=float("inf"))
    assert (n_acc == 3).all() and (path[:, :4] == [0, 1, 3, 5]).all() and (path[:, 4:] == -1).all()


def test_relaxed_accepts_more_as_delta_grows():
    rng = np.random.default_rng(33)
    B, R, V = 32, 9, 200
    logits = (rng.standard_normal((B, R, V)) * 2).astype(np.float32)
    tok = rng.integers(0, V, size=(B, R)).astype(np.int32)
    prev = None
    for delta in (0.0, 0.5, 1.0, 2.0, 4.0, 8.0, 1e9):
        n_acc, _, _ = oracle.accept_greedy_relaxed(logits, tok, delta=delta)
        if prev is not None:
            assert (n_acc >= prev).all()
        prev = n_acc
    assert prev.min() == R - 1


def test_relaxed_zero_delta_accepts_any_tied_maximum():
    # ids 1 and 3 tie for row 0's maximum: greedy wants id 1 (lowest index),
    # the relaxed test only the gap, which is 0 for either
    logits = np.zeros((1, 2, 5), np.float32)
    logits[0, 0, 1] = logits[0, 0, 3] = 2.0
    logits[0, 1, 4] = 1.0
    tok = np.array([[0, 3]], np.int32)
    assert int(oracle.accept_greedy(logits, tok)[0][0]) == 0
    n_acc, out_tok, path = oracle.accept_greedy_relaxed(logits, tok, delta=0.0)
    assert (int(n_acc[0]), int(out_tok[0]), path[0].tolist()) == (1, 4, [0, 1])


def test_relaxed_rejects_bad_inputs():
    logits = np.zeros((1, 3, 4), np.float32)
    tok = np.array([[0, 1, 1]], np.int32)
    for bad in (-0.1, float("nan")):
        with pytest.raises(oracle.OracleError):
            oracle.accept_greedy_relaxed(logits, tok, delta=bad)
    with pytest.raises(oracle.OracleError):
        oracle.accept_greedy_relaxed(logits, np.array([[0, 9, 0]], np.int32), delta=1.0)

def test_greedy_alignment_golden():
    g = json.load(open(os.path.join(GOLDEN, "alignment.json")))
    for case in g["cases"]:
        logits = np.array(case["logits"], np.float32)[None]
        tok = np.array(case["tok"], np.int32)[None]
        n_acc, out_tok, path = oracle.accept_greedy(logits, tok)
        assert n_acc[0] == case["n_acc"], case["why"]
        assert out_tok[0] == case["out_tok"], case["why"]
        assert path[0].tolist() == case["path"], case["why"]


def _random_greedy_case(rng, B, R, V, rate=0.6):
    logits = rng.standard_normal((B, R, V)).astype(np.float32)
    g = logits.argmax(-1)
    tok = rng.integers(0, V, size=(B, R)).astype(np.int32)
    plant = rng.random((B, R)) < rate
    tok[:, 1:] = np.where(plant[:, 1:], g[:, :-1], tok[:, 1:])
    return logits, tok


def test_greedy_chain_equals_single_child_tree():
    rng = np.random.default_rng(11)
    B, R, V = 64, 9, 50
    logits, tok = _random_greedy_case(rng, B, R, V, rate=0.8)
    parent = np.tile(np.arange(-1, R - 1, dtype=np.int32), (B, 1))
    a = oracle.accept_greedy(logits, tok)
    b = oracle.accept_greedy(logits, tok, parent)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert set(a[0].tolist()) > {0, R - 1}  # both ends occur


def test_greedy_tree_takes_first_matching_child_in_index_order():
    # root 0 with children 1, 2 (both carry the root's argmax 3); 2 has child 3.
    V = 6
    logits = np.zeros((1, 4, V), np.float32)
    logits[0, 0, 3] = 1.0
    logits[0, 1, 4] = 1.0
    logits[0, 2, 5] = 1.0
    logits[0, 3, 2] = 1.0
    parent = np.array([[-1, 0, 0, 2]], np.int32)
    tok = np.array([[0, 3, 3, 5]], np.int32)
    n_acc, out_tok, path = oracle.accept_greedy(logits, tok, parent)
    # node 1 wins over node 2 (index order), node 1 is a leaf -> bonus argmax of row 1
    assert (n_acc[0], out_tok[0], path[0].tolist()) == (1, 4, [0, 1, -1, -1])
    tok = np.array([[0, 1, 3, 5]], np.int32)
    n_acc, out_tok, path = oracle.accept_greedy(logits, tok, parent)
    assert (n_acc[0], out_tok[0], path[0].tolist()) == (2, 2, [0, 2, 3, -1])


def test_greedy_rejects_bad_inputs():
    logits = np.zeros((1, 3, 4), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.accept_greedy(logits, np.array([[0, 9, 0]], np.int32))
    with pytest.raises(oracle.OracleError):
        oracle.accept_greedy(logits, np.array([[0, 1, 1]], np.int32), np.array([[-1, 1, 0]], np.int32))


def test_sampling_reduces_to_greedy_at_one_hot():
    # p one-hot at the argmax (exp of -200 underflows to 0) and q one-hot at the
    # draft: a draft is accepted iff it equals the argmax, the residual is the
    # one-hot argmax, so sampling returns exactly the greedy decision.
    rng = np.random.default_rng(12)
    B, R, V = 200, 6, 32
    g = rng.integers(0, V, size=(B, R))
    logits = np.zeros((B, R, V), np.float32)
    np.put_along_axis(logits, g[..., None], 200.0, axis=-1)
    tok = rng.integers(0, V, size=(B, R)).astype(np.int32)
    plant = rng.random((B, R)) < 0.7
    tok[:, 1:] = np.where(plant[:, 1:], g[:, :-1], tok[:, 1:])
    q = np.zeros((B, R - 1, V), np.float32)
    np.put_along_axis(q, tok[:, 1:, None].astype(np.int64), 1.0, axis=-1)
    gs = oracle.accept_greedy(logits, tok)
    ss = oracle.accept_sample(logits, q, tok, seed=99, step=3)
    for x, y in zip(gs, ss):
        assert np.array_equal(x, y)


def test_sample_q_equal_p_always_accepts():
    rng = np.random.default_rng(13)
    B, R, V = 50, 5, 40
    logits = rng.standard_normal((B, R, V)).astype(np.float32)
    q = np.stack([np.stack([oracle.softmax(logits[b, u]) for u in range(R - 1)]) for b in range(B)])
    tok = rng.integers(0, V, size=(B, R)).astype(np.int32)
    n_acc, _, path = oracle.accept_sample(logits, q, tok, seed=5)
    assert np.all(n_acc == R - 1)
    assert np.all(path == np.arange(R))


def test_sample_disjoint_support_always_rejects_and_resamples_p():
    B, R, V = 64, 3, 8
    logits = np.full((B, R, V), -300.0, np.float32)
    logits[:, :, :4] = np.random.default_rng(1).standard_normal((B, R, 4)).astype(np.float32)
    q = np.zeros((B, R - 1, V), np.float32)
    q[:, :, 4:] = 0.25
    tok = np.full((B, R), 5, np.int32)
    n_acc, out_tok, _ = oracle.accept_sample(logits, q, tok, seed=8)
    assert np.all(n_acc == 0)
    assert np.all(out_tok < 4)   # the residual max(0, p - q) is p itself


def test_sample_chain_equals_single_child_tree():
    rng = np.random.default_rng(14)
    B, R, V = 40, 9, 300
    logits = (rng.standard_normal((B, R, V)) * 2).astype(np.float32)
    qlog = logits[:, :R - 1] + rng.standard_normal((B, R - 1, V)).astype(np.float32)
    q = np.exp(qlog - qlog.max(-1, keepdims=True))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    tok = np.zeros((B, R), np.int32)
    for b in range(B):
        for j in range(1, R):
            pr = q[b, j - 1].astype(np.float64)
            tok[b, j] = rng.choice(V, p=pr / pr.sum())
    parent = np.tile(np.arange(-1, R - 1, dtype=np.int32), (B, 1))
    q_tree = np.concatenate([q, np.zeros((B, 1, V), np.float32)], axis=1)
    for T in (1.0, 0.6):
        a = oracle.accept_sample(logits, q, tok, temperature=T, seed=2024, step=17)
        b = oracle.accept_sample(logits, q_tree, tok, parent, temperature=T, seed=2024, step=17)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_sample_vocab_padding_of_q():
    # [mini-infer, cross-device alignment]: q over a shorter draft vocab is
    # zero-padded; a token beyond it has q = 0 and is accepted, ids inside it
    # are unaffected by the padding.
    rng = np.random.default_rng(15)
    B, R, V, Vq = 30, 4, 64, 56
    logits = rng.standard_normal((B, R, V)).astype(np.float32)
    q = rng.random((B, R - 1, Vq)).astype(np.float32)
    q /= q.sum(-1, keepdims=True)
    tok = rng.integers(0, Vq, size=(B, R)).astype(np.int32)
    q_full = np.concatenate([q, np.zeros((B, R - 1, V - Vq), np.float32)], axis=-1)
    a = oracle.accept_sample(logits, q, tok, seed=1)
    b = oracle.accept_sample(logits, q_full, tok, seed=1)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    tok[:, 1] = V - 1
    n_acc, _, _ = oracle.accept_sample(logits, q, tok, seed=1)
    assert np.all(n_acc >= 1)


def test_sample_philox_matches_injected_uniforms():
    # The Philox stream (key = seed, counter = (b, node, step)) and the same
    # values passed in explicitly give identical results.
    rng = np.random.default_rng(16)
    B, R, V = 20, 6, 100
    logits = rng.standard_normal((B, R, V)).astype(np.float32)
    q = rng.random((B, R - 1, V)).astype(np.float32)
    q /= q.sum(-1, keepdims=True)
    tok = rng.integers(0, V, size=(B, R)).astype(np.int32)
    seed, step = 0x1234_5678_9ABC, 77
    uni = np.zeros((B, R, 2), np.float32)
    for b in range(B):
        for u in range(R):
            w = oracle.philox4x32_10([b, u, step & 0xFFFFFFFF, step >> 32], [seed & 0xFFFFFFFF, seed >> 32])
            uni[b, u] = [oracle.uniform24(w[0]), oracle.uniform24(w[1])]
    a = oracle.accept_sample(logits, q, tok, seed=seed, step=step)
    b_ = oracle.accept_sample(logits, q, tok, uniforms=uni)
    for x, y in zip(a, b_):
        assert np.array_equal(x, y)


# ----------------------------------------------------------------------------
# exact enumeration on a 5-token vocab
# ----------------------------------------------------------------------------

V5 = 5
Q5 = np.array([0.5, 0.25, 0.125, 0.0625, 0.0625], np.float32)   # sums to 1 exactly
L5 = np.array([0.3, -1.2, 1.1, 0.4, -0.5], np.float32)          # target logits


def _filled(block, n, dtype):
    out = np.empty((n,) + np.shape(block), dtype)
    out[...] = block
    return out


def _sweep(logits_row_block, q_block, tok_row, parent_row, vary, fixed_u, chunk=1 << 21):
    """Run the oracle over all 2^24 grid values of one uniform.
    vary = (node, word); fixed_u [R, 2] supplies the others.  Returns
    (n_acc, path[:, 1], out_tok) over the grid."""
    R = logits_row_block.shape[0]
    node, word = vary
    logits = _filled(logits_row_block, chunk, np.float32)
    q = _filled(q_block, chunk, np.float32)
    tok = _filled(tok_row, chunk, np.int32)
    par = None if parent_row is None else _filled(parent_row, chunk, np.int32)
    uni = _filled(fixed_u, chunk, np.float32)
    grid = np.arange(chunk, dtype=np.float64)
    res_n, res_p1, res_tok = [], [], []
    for start in range(0, GRID, chunk):
        uni[:, node, word] = ((grid + start) * 2.0 ** -24).astype(np.float32)
        n_acc, out_tok, path = oracle.accept_sample(logits, q, tok, par, uniforms=uni)
        res_n.append(n_acc)
        res_p1.append(path[:, 1].copy())
        res_tok.append(out_tok)
    return np.concatenate(res_n), np.concatenate(res_p1), np.concatenate(res_tok)


def _frac_vec(x):
    return [Fraction(float(v)) for v in x]


@pytest.mark.slow
def test_enumeration_chain_single_position_equals_p():
    p = oracle.softmax(L5)
    logits = np.stack([L5, np.zeros(V5, np.float32)])      # row 0 verifies d1; row 1 = bonus row
    q = Q5[None]
    fixed = np.array([[0.5, 0.5], [0.5, 0.5]], np.float32)
    acc = []
    for d in range(V5):
        n_acc, _, _ = _sweep(logits, q, np.array([0, d], np.int32), None, (1, 0), fixed)
        acc.append(int(n_acc.sum()))
    # forced rejection: a token with p < q, u_acc at the top of the grid
    d_rej = int(np.argmin(p / Q5))
    assert p[d_rej] / Q5[d_rej] < 1 - 2.0 ** -23
    fixed_rej = np.array([[0.5, 0.5], [U_MAX, 0.5]], np.float32)
    n_acc, _, out = _sweep(logits, q, np.array([0, d_rej], np.int32), None, (0, 1), fixed_rej)
    assert np.all(n_acc == 0)
    res = np.bincount(out, minlength=V5)
    qf, pf = _frac_vec(Q5), _frac_vec(p)
    P = [sum(qf[d] * (Fraction(acc[d], GRID) * (x == d) + (1 - Fraction(acc[d], GRID)) * Fraction(int(res[x]), GRID))
             for d in range(V5)) for x in range(V5)]
    # grid quantisation of each threshold (< 2^-24 per token) and float
    # rounding of p, the residual and its sums (a few ulp of 1) bound the gap
    for x in range(V5):
        assert abs(float(P[x] - pf[x])) <= 6 * 2.0 ** -24, (x, float(P[x]), float(pf[x]))
    # the accept counts are exactly the grid points below min(1, p/q)
    for d in range(V5):
        r = float(np.float32(p[d]) / np.float32(Q5[d]))
        assert acc[d] == min(GRID, int(np.ceil(r * GRID)))


def _tree_enumeration(b_children):
    R = 1 + b_children
    parent = np.array([-1] + [0] * b_children, np.int32)
    p = oracle.softmax(L5)
    logits = np.zeros((R, V5), np.float32)
    logits[0] = L5
    q = np.zeros((R, V5), np.float32)
    q[0] = Q5
    d_rej = int(np.argmin(p / Q5))   # p < q there: rejectable at stage 0 and zero in every residual
    base_u = np.full((R, 2), 0.5, np.float32)
    base_u[1:, 0] = U_MAX              # children rejected unless swept
    A = []                              # A[i][x]: accept count of child i+1 carrying token x
    for i in range(b_children):
        row = []
        for x in range(V5):
            tok = np.array([0] + [d_rej] * b_children, np.int32)
            tok[1 + i] = x
            _, p1, _ = _sweep(logits, q, tok, parent, (1 + i, 0), base_u)
            row.append(int(np.sum(p1 == 1 + i)))
            # children before the swept one were all rejected
            assert not np.any((p1 >= 1) & (p1 < 1 + i))
        A.append(row)
    tok = np.array([0] + [d_rej] * b_children, np.int32)
    n_acc, _, out = _sweep(logits, q, tok, parent, (0, 1), base_u)
    assert np.all(n_acc == 0)
    res = np.bincount(out, minlength=V5)
    qf = _frac_vec(Q5)
    P = [Fraction(int(res[x]), GRID) for x in range(V5)]      # after the last child
    for i in reversed(range(b_children)):
        a = [Fraction(A[i][y], GRID) for y in range(V5)]
        P = [sum(qf[y] * (a[y] * (x == y) + (1 - a[y]) * P[x]) for y in range(V5)) for x in range(V5)]
    return P, _frac_vec(p)


@pytest.mark.slow
@pytest.mark.parametrize("b_children", [2, 3])
def test_enumeration_tree_siblings_equals_p(b_children):
    P, pf = _tree_enumeration(b_children)
    for x in range(V5):
        assert abs(float(P[x] - pf[x])) <= 8 * 2.0 ** -24 * b_children, (x, float(P[x]), float(pf[x]))


def _exact_recursive_rejection(p, q, n_children):
    """The algorithm in exact rationals: P_i = min(q, w_i) + (1 - sum min(q, w_i)) P_{i+1},
    w_{i+1} = norm(max(0, w_i - q)), P_n = w_n."""
    w = list(p)
    stages = []
    for _ in range(n_children):
        mn = [min(a, b) for a, b in zip(q, w)]
        beta = sum(mn)
        stages.append((mn, beta))
        rho = [max(Fraction(0), a - b) for a, b in zip(w, q)]
        S = sum(rho)
        w = [r / S for r in rho] if S > 0 else w
    P = w
    for mn, beta in reversed(stages):
        P = [m + (1 - beta) * x for m, x in zip(mn, P)]
    return P


def test_exact_rational_algorithm_preserves_p():
    p = [Fraction(n, 20) for n in (1, 7, 3, 5, 4)]
    q = [Fraction(n, 16) for n in (8, 4, 2, 1, 1)]
    for k in (1, 2, 3, 4):
        assert _exact_recursive_rejection(p, q, k) == p
