"""Shared helpers for the -m gpu parity tests: tolerances and comparisons against the oracle."""
import numpy as np
import torch

# Tolerances against the fp64 oracle on identical (dtype-rounded) inputs:
#   fp32 path: max abs error <= 1e-4 on o
#   bf16 path: max abs error <= 2e-2 and mean abs error <= 2e-3 on o
F32_MAX = 1e-4
BF16_MAX = 2e-2
BF16_MEAN = 2e-3
LSE_F32_MAX = 1e-4
LSE_BF16_MAX = 2e-2


def to_np(t: torch.Tensor):
    return t.detach().to("cpu", torch.float64).numpy()


def check(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), what + ": non-finite output"
    err = np.abs(got - ref)
    mx, mean = float(err.max()), float(err.mean())
    if dtype == torch.float32:
        assert mx <= F32_MAX, "%s: max abs err %.3g > %.1g" % (what, mx, F32_MAX)
    else:
        assert mx <= BF16_MAX, "%s: max abs err %.3g > %.1g" % (what, mx, BF16_MAX)
        assert mean <= BF16_MEAN, "%s: mean abs err %.3g > %.1g" % (what, mean, BF16_MEAN)
    return mx, mean


def check_lse(got, ref, dtype, what=""):
    err = float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))))
    tol = LSE_F32_MAX if dtype == torch.float32 else LSE_BF16_MAX
    assert err <= tol, "%s: lse max abs err %.3g > %.1g" % (what, err, tol)
    return err


def cuda(x):
    return None if x is None else x.cuda()
