"""Shared helpers of the GPU parity tests: host copies for the oracle and the tolerance checks.

Tolerances: index scores and top-k lists are compared bit-for-bit; attention outputs must be
within max-abs 1e-2 and relative L2 5e-3 of the fp64 oracle; compressed entries (bf16) within
one bf16 rounding (2^-8 relative) plus 1e-6 absolute of the fp64 pooled value."""
import numpy as np
import torch

import oracle as O

ATT_MAX_ABS = 1e-2
ATT_REL_L2 = 5e-3
LSE_ABS = 2e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return O.bf16_to_f64(bits(t))
    return t.detach().cpu().numpy().astype(np.float64)


def npy(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_attention_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / denom if denom > 0 else float(np.linalg.norm(got))
    assert max_abs <= ATT_MAX_ABS and rel <= ATT_REL_L2, \
        f"{what}: max_abs={max_abs:.3e} rel_l2={rel:.3e}"


def assert_lse_close(got: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    inf_g, inf_r = np.isneginf(got), np.isneginf(ref)
    assert np.array_equal(inf_g, inf_r), what
    fin = ~inf_r
    if fin.any():
        assert np.max(np.abs(got[fin] - ref[fin])) <= LSE_ABS, what


def assert_entries_close(got_bits: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    got = O.bf16_to_f64(got_bits)
    tol = np.abs(ref) * 2.0 ** -8 + 1e-6
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} entries off, worst " \
                          f"{float(np.max(np.abs(got - ref) - tol)):.3e}"
