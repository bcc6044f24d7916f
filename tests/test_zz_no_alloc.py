"""sv_accept_sample_noalloc: the sampled acceptance for callers that cannot
allocate device memory (a plugin handed only its buffers, a loop that must
not allocate).  It must return exactly what sv_accept_sample returns for the
same inputs, call after call, although its scratch is one fixed device array
that every call reuses.

Kept in its own file so that pytest collects it after every other test."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_sv_gb300 import synth

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


def test_noalloc_rejects_rows_beyond_the_fixed_scratch(sv):
    B, R, V = 8193, 1, 16
    logits = torch.zeros(B, R, V, device="cuda")
    q = torch.zeros(B, 0, V, device="cuda")
    tok = torch.zeros(B, R, dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SVError) as e:
        sv.accept_sample_noalloc(logits, q, tok)
    assert e.value.status == 2
