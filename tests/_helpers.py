"""Small helpers shared by the GPU parity tests."""
import numpy as np
import torch

from speculative_decoding_verification_sv_gb300 import synth


def bits(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_bits(t)


def np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def within_tol(got: np.ndarray, ref: np.ndarray, frac: float = 1e-2):
    """The float parity bar: max|got - ref| <= frac * max|ref|."""
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    bound = frac * float(np.max(np.abs(ref)))
    return err <= bound, err, bound


def assert_same(gpu_outputs, oracle_outputs, what=""):
    for i, (a, b) in enumerate(zip(gpu_outputs, oracle_outputs)):
        a = a.detach().cpu().numpy() if isinstance(a, torch.Tensor) else np.asarray(a)
        if not np.array_equal(a, b):
            bad = np.argwhere(a != b)[:5]
            raise AssertionError(f"{what} output {i} differs at {bad.tolist()}: gpu {a[tuple(bad[0])]} "
                                 f"oracle {b[tuple(bad[0])]}")
