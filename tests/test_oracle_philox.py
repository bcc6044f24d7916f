"""Pins for the oracle's Philox4x32-10 stream and its uniform construction.

Philox4x32-10 is fixed by its publication (Salmon, Moraes, Dror, Shaw, SC'11);
the pages only name the generator, with key = seed and counter = (sequence,
position).  The oracle is checked against
  * Triton's independent Philox implementation, run on the CPU through the
    Triton interpreter (key = seed, counter = (offset, 0, 0, 0)), and
  * an inverse written here from the round function's definition: each round
    is a bijection whose multiplications can be undone with the modular
    inverses of the two multipliers, so decrypting the oracle's output with
    the published constants must give back the counter.
"""
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

import oracle

M_A, M_B = 0xD2511F53, 0xCD9E8D57
W_A, W_B = 0x9E3779B9, 0xBB67AE85
MASK = 0xFFFFFFFF


def _inverse(out, key):
    """Undo ten Philox4x32 rounds.  Forward round with key (k0, k1):
    y0 = hi(B*x2) ^ x1 ^ k0, y1 = lo(B*x2), y2 = hi(A*x0) ^ x3 ^ k1, y3 = lo(A*x0)."""
    inv_a = pow(M_A, -1, 1 << 32)
    inv_b = pow(M_B, -1, 1 << 32)
    keys = []
    k0, k1 = key
    for r in range(10):
        keys.append((k0, k1))
        k0 = (k0 + W_A) & MASK
        k1 = (k1 + W_B) & MASK
    y0, y1, y2, y3 = (int(v) for v in out)
    for k0, k1 in reversed(keys):
        x0 = (y3 * inv_a) & MASK
        x2 = (y1 * inv_b) & MASK
        hi_a = (M_A * x0) >> 32
        hi_b = (M_B * x2) >> 32
        x1 = y0 ^ hi_b ^ k0
        x3 = y2 ^ hi_a ^ k1
        y0, y1, y2, y3 = x0, x1, x2, x3
    return [y0, y1, y2, y3]


def test_inverse_recovers_counter():
    rng = np.random.default_rng(1)
    for _ in range(2000):
        ctr = [int(v) for v in rng.integers(0, 2**32, size=4, dtype=np.uint64)]
        key = [int(v) for v in rng.integers(0, 2**32, size=2, dtype=np.uint64)]
        out = oracle.philox4x32_10(ctr, key)
        assert _inverse(out, key) == ctr


def test_distinct_counters_distinct_outputs():
    seen = set()
    for b in range(16):
        for u in range(16):
            seen.add(tuple(oracle.philox4x32_10([b, u, 7, 0], [123, 456])))
    assert len(seen) == 256


_TRITON_SCRIPT = textwrap.dedent(r"""
    import os, sys, json
    os.environ["TRITON_INTERPRET"] = "1"
    import numpy as np, torch, triton, triton.language as tl

    @triton.jit
    def k(out_ptr, seed, off_ptr, N: tl.constexpr):
        i = tl.arange(0, N)
        offs = tl.load(off_ptr + i)
        a, b, c, d = tl.randint4x(seed, offs)
        tl.store(out_ptr + i * 4 + 0, a)
        tl.store(out_ptr + i * 4 + 1, b)
        tl.store(out_ptr + i * 4 + 2, c)
        tl.store(out_ptr + i * 4 + 3, d)

    cases = json.loads(sys.argv[1])
    res = []
    for seed, offs in cases:
        o = torch.tensor(offs, dtype=torch.int32)
        out = torch.zeros(len(offs) * 4, dtype=torch.int32)
        k[(1,)](out, seed, o, N=len(offs))
        res.append((out.numpy().view(np.uint32).reshape(-1, 4)).tolist())
    print(json.dumps(res))
""")


def test_matches_triton_interpreter():
    pytest.importorskip("triton")
    import json
    rng = np.random.default_rng(7)
    cases = []
    for _ in range(6):
        seed = int(rng.integers(1, 2**62))
        offs = [int(v) for v in rng.integers(0, 2**31 - 1, size=16)]
        cases.append((seed, offs))
    env = dict(os.environ, TRITON_INTERPRET="1")
    r = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT, json.dumps(cases)], capture_output=True,
                       text=True, env=env, timeout=600)
    if r.returncode != 0:
        pytest.skip("triton interpreter unavailable: " + r.stderr[-300:])
    got = json.loads(r.stdout.strip().splitlines()[-1])
    for (seed, offs), rows in zip(cases, got):
        key = [seed & MASK, seed >> 32]
        for off, row in zip(offs, rows):
            assert list(oracle.philox4x32_10([off, 0, 0, 0], key)) == row


def test_uniform24_grid():
    assert oracle.uniform24(0) == 0.0
    assert oracle.uniform24(0xFF) == 0.0
    assert oracle.uniform24(0x100) == 2.0 ** -24
    assert oracle.uniform24(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    assert oracle.uniform24(0x80000000) == 0.5
