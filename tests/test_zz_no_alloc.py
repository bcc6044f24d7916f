"""sv_accept_sample_noalloc: the sampled acceptance for callers that cannot
allocate device memory (a plugin handed only its buffers, a loop that must
not allocate).  It must return exactly what sv_accept_sample returns, and
what the oracle computes, for the same inputs, call after call, although its
scratch is one fixed device array that every call reuses.

Kept in its own file so that pytest collects it after every other test."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_sv_gb300 import synth

from _helpers import assert_same

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_sv_gb300 import binding
    return binding


def _same(a, b):
    for x, y in zip(a, b):
        assert torch.equal(x, y), (x, y)


def test_noalloc_matches_workspace_entry_on_consecutive_calls(sv):
    # two different rounds back to back: the second call must not see stale
    # statistics from the first
    cases = [synth.sample_inputs(64, 8, 151936, wid=2),
             synth.sample_inputs(16, 5, 32768, wid=130, logit_std=1.5)]
    for i, si in enumerate(cases):
        args = (si.logits.cuda(), si.q.cuda(), si.tok.cuda())
        ref = sv.accept_sample(*args, seed=77 + i, step=i)
        got = sv.accept_sample_noalloc(*args, seed=77 + i, step=i)
        torch.cuda.synchronize()
        _same(got, ref)
    assert sv.get_device_error() == 0


def test_noalloc_tree_and_injected_uniforms(sv):
    par = synth.random_tree(20, 5, 3, 4)
    si = synth.sample_inputs(6, len(par) - 1, 8192, wid=131, parent=par, logit_std=1.0)
    rng = np.random.default_rng(5)
    for _ in range(2):
        uni = torch.from_numpy((rng.integers(0, 2 ** 24, size=(6, len(par), 2)) * 2.0 ** -24).astype(np.float32))
        args = (si.logits.cuda(), si.q.cuda(), si.tok.cuda(), si.parent.cuda())
        _same(sv.accept_sample_noalloc(*args, uniforms=uni.cuda()), sv.accept_sample(*args, uniforms=uni.cuda()))


def test_noalloc_matches_oracle_chain_b64(sv):
    # the full-size sampled workload, checked against the oracle directly (not
    # only against the other GPU entry point), twice in a row
    si = synth.sample_inputs(64, 8, 151936, wid=2)
    exp = oracle.accept_sample(si.logits.numpy(), si.q.numpy(), si.tok.numpy(), seed=2024, step=7)
    args = (si.logits.cuda(), si.q.cuda(), si.tok.cuda())
    for _ in range(2):
        assert_same(sv.accept_sample_noalloc(*args, seed=2024, step=7), exp, "noalloc chain b64")
    assert sv.get_device_error() == 0


def test_noalloc_matches_oracle_tree_full_vocab(sv):
    # a 64-node depth-8 draft tree at the 7B vocabulary, draft vocab smaller
    par = synth.random_tree(64, 8, 3, 40)
    si = synth.sample_inputs(2, len(par) - 1, 152064, wid=132, Vq=151936, logit_std=1.5, parent=par)
    args = (si.logits.cuda(), si.q.cuda(), si.tok.cuda(), si.parent.cuda())
    for step in (0, 3):
        exp = oracle.accept_sample(si.logits.numpy(), si.q.numpy(), si.tok.numpy(), si.parent.numpy(), seed=11,
                                   step=step)
        assert_same(sv.accept_sample_noalloc(*args, seed=11, step=step), exp, f"noalloc tree step {step}")
    assert sv.get_device_error() == 0


@pytest.mark.parametrize("B", [1, 2, 3])
def test_noalloc_small_chains(sv, B):
    # chains of one to three sequences take the same cluster walk as larger ones
    si = synth.sample_inputs(B, 4, 151936, wid=133 + B)
    args = (si.logits.cuda(), si.q.cuda(), si.tok.cuda())
    exp = oracle.accept_sample(si.logits.numpy(), si.q.numpy(), si.tok.numpy(), seed=5, step=B)
    got = sv.accept_sample_noalloc(*args, seed=5, step=B)
    assert_same(got, exp, f"noalloc chain B={B}")
    _same(got, sv.accept_sample(*args, seed=5, step=B))


def test_noalloc_rejects_rows_beyond_the_fixed_scratch(sv):
    B, R, V = 8193, 1, 16
    logits = torch.zeros(B, R, V, device="cuda")
    q = torch.zeros(B, 0, V, device="cuda")
    tok = torch.zeros(B, R, dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SVError) as e:
        sv.accept_sample_noalloc(logits, q, tok)
    assert e.value.status == 2
