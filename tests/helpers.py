"""Shared helpers for the parity tests (tolerances, conversions, near-tie logic)."""
import numpy as np
import torch

# Scores (rule_j, R_b, M_t): relative 1e-3 with an absolute floor of 1e-6 * max|ref|.
SCORE_RTOL = 1e-3
SCORE_FLOOR = 1e-6
# Near-tie band for integer decisions made from floating point scores.
TIE_RTOL = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def assert_scores_close(got, ref, rtol=SCORE_RTOL, floor=SCORE_FLOOR, what="scores"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    tol = rtol * np.abs(ref) + floor * max(np.abs(ref).max(initial=0.0), 1e-300)
    err = np.abs(got - ref)
    bad = np.flatnonzero(err > tol)
    assert bad.size == 0, (f"{what}: {bad.size} of {ref.size} outside rel {rtol}; worst at {bad[np.argmax(err[bad])]}:"
                           f" got {got.flat[bad[0]]!r} ref {ref.flat[bad[0]]!r}")


def bf16_ulp(v):
    """Spacing of bf16 values at |v| (float32 spacing * 2^16)."""
    v = np.abs(np.asarray(v, np.float64)).astype(np.float32)
    return np.spacing(np.maximum(v, np.float32(2.0 ** -126))).astype(np.float64) * 2.0 ** 16


def assert_keep_sets_match(got_idx, ref_idx, ref_score, kth_score, forced, what="keep set"):
    """Kept sets equal except for candidates whose oracle score lies within
    TIE_RTOL (relative) of the oracle's k-th kept score."""
    got, ref = set(np.asarray(got_idx).tolist()), set(np.asarray(ref_idx).tolist())
    assert len(got) == len(ref), f"{what}: sizes differ {len(got)} vs {len(ref)}"
    diff = got ^ ref
    band = TIE_RTOL * abs(kth_score) + 1e-30
    for j in diff:
        assert not forced(j), f"{what}: forced position {j} differs"
        assert abs(ref_score[j] - kth_score) <= band, (
            f"{what}: position {j} differs with score {ref_score[j]!r}, k-th score {kth_score!r}")
