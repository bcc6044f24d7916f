"""The library's once-per-device set-up (kernel attributes, cached device
addresses) is shared by every host thread: calls made from two threads at once,
each on its own stream and buffers, give the oracle's results."""
import threading

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_sv_gb300 import synth

from _helpers import assert_same

pytestmark = pytest.mark.gpu


def test_two_threads_sampled_and_greedy():
    from speculative_decoding_verification_sv_gb300 import binding as sv
    cases = [synth.sample_inputs(8, 4, 151936, wid=140 + i, logit_std=2.0) for i in range(2)]
    exp = [oracle.accept_sample(c.logits.numpy(), c.q.numpy(), c.tok.numpy(), seed=9, step=i)
           for i, c in enumerate(cases)]
    rng = np.random.default_rng(4)
    glog = [rng.standard_normal((4, 5, 50000)).astype(np.float32) for _ in range(2)]
    gtok = [synth.plant_chain_drafts(g.argmax(-1), 0.6, 50000, seed=i) for i, g in enumerate(glog)]
    gexp = [oracle.accept_greedy(g, t) for g, t in zip(glog, gtok)]
    got, errors = [None, None], []

    def work(i):
        try:
            torch.cuda.set_device(0)
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                res = []
                for _ in range(20):   # many calls, so the two threads overlap
                    c = cases[i]
                    a = sv.accept_sample(c.logits.cuda(), c.q.cuda(), c.tok.cuda(), seed=9, step=i, stream=st)
                    b = sv.accept_greedy(torch.from_numpy(glog[i]).cuda(), torch.from_numpy(gtok[i]).cuda(),
                                         stream=st)
                    res.append((a, b))
                st.synchronize()
                got[i] = res
        except Exception as e:   # pragma: no cover - reported below
            errors.append(e)

    ths = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in ths:
        t.start()
    for t in ths:
        t.join()
    assert not errors, errors
    for i in range(2):
        for a, b in got[i]:
            assert_same(a, exp[i], f"thread {i} sampled")
            assert_same(b, gexp[i], f"thread {i} greedy")
    assert sv.get_device_error() == 0
