"""GPU parity of the sampled acceptance's building blocks, through the C ABI's
diagnostic entry points: the device exponential, Philox4x32-10 and the
canonical summation tree with its descent sampler must equal the oracle's
independent implementations bit for bit."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_sv_gb300 import binding
    return binding


def test_exp_bit_exact_dense(sv):
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        np.linspace(-105.0, 0.0, 2_000_001, dtype=np.float32),
        rng.uniform(-104.0, 0.0, 2_000_000).astype(np.float32),
        -np.abs(rng.standard_normal(500_000).astype(np.float32)) * 1e-3,
        np.array([0.0, -0.0, -1e-30, -87.3, -88.0, -103.99, -104.0, -104.01, -np.inf, np.nan], np.float32),
        # around the lower end of the normal-range form (-86.5) and its k = -125
        np.nextafter(np.float32(-86.5), np.float32(0), dtype=np.float32)[None],
        np.array([-86.5, -86.49, -86.0, -86.64, -86.65, -86.99, -87.0], np.float32),
    ])
    got = sv.diag_exp(torch.from_numpy(xs).cuda()).cpu().numpy()
    ref = oracle.exp32_array(xs)
    same = (got.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), xs[~same][:5]


def test_division_bit_exact(sv):
    """The acceptance divides by a row's sum Z (in [1, V]) and by sibling
    residual sums S (in (0, 1]) through a reciprocal and one correction step;
    its quotients must be IEEE float32 division rounded to nearest, which
    numpy computes on the host."""
    rng = np.random.default_rng(5)
    n = 4_000_000

    def f32(lo_exp, hi_exp, size):   # random significands, exponents uniform in [lo, hi]
        e = rng.integers(lo_exp, hi_exp + 1, size=size)
        m = rng.integers(0, 2 ** 23, size=size)
        return ((e + 127).astype(np.uint32) << 23 | m.astype(np.uint32)).view(np.float32)

    # divisors with special significands (1, all ones, 1 + ulp, 1.5, ...)
    sig = np.array([0, 0x7FFFFF, 1, 0x400000, 0x7FFFFE, 0x3FFFFF, 0x555555], np.uint32)
    bexp = np.array([0, 1, 5, 12, 17, -1, -7, -40], np.int64)
    bs = ((bexp[:, None] + 127).astype(np.uint32) << 23 | sig[None, :]).view(np.float32).ravel()
    a_dense = (np.uint32(0x3F000000) | np.arange(0, 2 ** 23, 64, dtype=np.uint32)).view(np.float32)
    pairs = [
        (np.tile(a_dense, bs.size), np.repeat(bs, a_dense.size)),
        (f32(-59, -1, n), f32(0, 17, n)),                          # e / Z
        (f32(-50, -1, n), f32(-50, -1, n)),                        # rho / S (any order of sizes)
        (f32(-60, 59, n), f32(-60, 59, n)),                        # the whole fast range
        (f32(-126, -61, 100_000), f32(0, 17, 100_000)),            # below it: the division itself
        (np.array([0.0, 1.0, 2.0 ** -60, 2.0 ** -61, 1e-45, 3.0, 1.0], np.float32),
         np.array([3.0, 3.0, 7.0, 7.0, 3.0, 2.0 ** -61, 2.0 ** 61], np.float32)),
    ]
    a = np.concatenate([p[0] for p in pairs]).astype(np.float32)
    b = np.concatenate([p[1] for p in pairs]).astype(np.float32)
    got = sv.diag_div(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()).cpu().numpy()
    ref = a / b
    same = got.view(np.uint32) == ref.view(np.uint32)
    assert same.all(), (a[~same][:5], b[~same][:5])


def test_philox_bit_exact(sv):
    rng = np.random.default_rng(2)
    n = 200_000
    ctr = rng.integers(0, 2 ** 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2 ** 32, size=(n, 2), dtype=np.uint64).astype(np.uint32)
    got = sv.diag_philox(torch.from_numpy(ctr.view(np.int32)).cuda(),
                         torch.from_numpy(key.view(np.int32)).cuda()).cpu().numpy().view(np.uint32)
    for i in range(0, n, 997):
        assert np.array_equal(got[i], oracle.philox4x32_10(ctr[i], key[i]))


@pytest.mark.parametrize("n", [4, 8, 100, 1000, 4096, 4100, 40000, 131072, 151936, 152064, 262144])
def test_canonical_sum_and_descent_bit_exact(sv, n):
    rng = np.random.default_rng(n)
    m = 24
    x = rng.exponential(size=(m, n)).astype(np.float32)
    x[::3, rng.integers(0, n, size=n // 3)] = 0.0                # sparse rows
    x[1, : n // 2] = 0.0                                        # mass only in the upper half
    x[2] *= np.float32(1e-30)                                   # tiny values
    u = rng.random(m).astype(np.float32)
    u[0] = 0.0
    u[4] = np.float32(1.0 - 2.0 ** -24)
    sums, draws = sv.diag_canon(torch.from_numpy(x).cuda(), torch.from_numpy(u).cuda())
    sums, draws = sums.cpu().numpy(), draws.cpu().numpy()
    for i in range(m):
        assert sums[i].view(np.uint32) == np.float32(oracle.canon_sum(x[i])).view(np.uint32), i
        assert draws[i] == oracle.tree_sample(x[i], float(u[i])), i
