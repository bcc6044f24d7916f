"""The seeded synthetic input generators hold to the recipe they state:
the draft tree's shape rules, the planted drafts' acceptance structure, the
sampled inputs' q rows, and reproducibility from the seed.  CPU only."""
import numpy as np
import torch

from speculative_decoding_verification_sv_gb300 import synth


def _children(parent):
    kids = [[] for _ in parent]
    for c in range(1, len(parent)):
        kids[parent[c]].append(c)
    return kids


def test_random_tree_shape_rules():
    for seed in range(6):
        par = synth.random_tree(64, 8, 3, seed)
        assert len(par) == 65 and par[0] == -1
        assert all(0 <= par[c] < c for c in range(1, 65))           # topological order
        d = synth.tree_depths(par)
        assert d.max() == 8                                         # the spine reaches depth 8, no deeper
        assert all(d[c] == d[par[c]] + 1 for c in range(1, 65))
        assert np.all(np.diff(d) >= 0)                              # breadth-first labels
        assert max(len(k) for k in _children(par)) <= 3
        assert np.array_equal(par, synth.random_tree(64, 8, 3, seed))   # reproducible
    assert not np.array_equal(synth.random_tree(64, 8, 3, 0), synth.random_tree(64, 8, 3, 1))


def test_plant_chain_drafts_structure():
    rng = np.random.default_rng(0)
    B, R, V = 400, 9, 1000
    g = rng.integers(0, V, size=(B, R))
    tok = synth.plant_chain_drafts(g, 0.55, V, seed=3)
    hit = tok[:, 1:] == g[:, :-1]
    assert 0.50 < hit.mean() < 0.60                                 # the planting rate
    assert ((tok >= 0) & (tok < V)).all()
    # a draft that is not planted is never the verifying row's argmax
    assert np.array_equal(synth.plant_chain_drafts(g, 0.0, V, seed=4)[:, 1:] != g[:, :-1],
                          np.ones((B, R - 1), bool))
    assert (synth.plant_chain_drafts(g, 1.0, V, seed=5)[:, 1:] == g[:, :-1]).all()


def test_plant_tree_drafts_follow_the_parent_row():
    rng = np.random.default_rng(1)
    par = synth.random_tree(20, 5, 3, 2)
    B, R, V = 30, len(par), 500
    g = rng.integers(0, V, size=(B, R))
    parent = np.tile(par, (B, 1))
    tok = synth.plant_tree_drafts(g, parent, 1.0, V, seed=6)
    for c in range(1, R):
        assert (tok[:, c] == g[:, par[c]]).all()
    tok0 = synth.plant_tree_drafts(g, parent, 0.0, V, seed=7)
    for c in range(1, R):
        assert (tok0[:, c] != g[:, par[c]]).all()


def test_sample_inputs_q_rows_are_distributions():
    si = synth.sample_inputs(6, 4, 3000, wid=5, Vq=2900)
    assert si.logits.shape == (6, 5, 3000) and si.q.shape == (6, 4, 2900)
    s = si.q.double().sum(-1)
    assert torch.allclose(s, torch.ones_like(s), atol=1e-5)
    assert (si.q >= 0).all()
    assert ((si.tok[:, 1:] >= 0) & (si.tok[:, 1:] < 2900)).all()   # drafts come from the draft vocab
    again = synth.sample_inputs(6, 4, 3000, wid=5, Vq=2900)
    assert torch.equal(si.logits, again.logits) and torch.equal(si.tok, again.tok)
    # trees: q has a row per node and the children of u are drawn from row u's support
    par = synth.random_tree(10, 4, 3, 1)
    st = synth.sample_inputs(3, len(par) - 1, 500, wid=6, parent=par)
    assert st.q.shape == (3, len(par), 500) and st.parent.shape == (3, len(par))
    for c in range(1, len(par)):
        assert (st.q[torch.arange(3), int(par[c]), st.tok[:, c].long()] > 0).all()


def test_bf16_bits_roundtrip():
    x = torch.randn(64).to(torch.bfloat16)
    b = synth.bf16_bits(x)
    assert b.dtype == np.uint16
    back = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16)
    assert torch.equal(back, x)
