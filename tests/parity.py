"""Shared parity helpers: compare the CUDA outputs with the fp64 oracle."""
import numpy as np
import torch

# Tolerances for fp16/bf16 inputs with fp32 accumulation.
O_TOL = 2e-2
LSE_TOL = 1e-3


def to_np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def compare(o_gpu, lse_gpu, o_ref, lse_ref, rows=None, o_tol=O_TOL, lse_tol=LSE_TOL):
    """o_gpu [b, sq, h, d], lse_gpu [b, h, sq] (device tensors); o_ref/lse_ref
    from the oracle for ``rows`` (all rows when None). Returns the errors."""
    o = to_np64(o_gpu)
    lse = to_np64(lse_gpu)
    if rows is not None:
        o = o[:, rows]
        lse = lse[:, :, rows]
    assert o.shape == o_ref.shape and lse.shape == lse_ref.shape
    assert np.all(np.isfinite(o)), "non-finite O"
    assert np.all(np.isfinite(lse)), "non-finite LSE"
    err_o = float(np.abs(o - o_ref).max())
    err_l = float(np.abs(lse - lse_ref).max())
    assert err_o <= o_tol, f"max |O - O_ref| = {err_o:.3e} > {o_tol}"
    assert err_l <= lse_tol, f"max |LSE - LSE_ref| = {err_l:.3e} > {lse_tol}"
    return err_o, err_l


def compare_masked(o_gpu, lse_gpu, o_ref, lse_ref, rows=None):
    """compare() for results in which some rows see no key (the causal mask
    with sq > sk): those rows must hold O = 0 and LSE = -inf exactly, as the
    oracle's -inf LSE marks them; the others are compared as usual.
    o_ref/lse_ref cover ``rows`` (all rows when None)."""
    sel = rows if rows is not None else list(range(o_gpu.shape[1]))
    seen = np.isfinite(lse_ref).all(axis=(0, 1))
    if (~seen).any():
        bad = [r for r, s_ in zip(sel, seen) if not s_]
        o64 = to_np64(o_gpu)[:, bad]
        l64 = to_np64(lse_gpu)[:, :, bad]
        assert np.all(o64 == 0.0), "a row with no visible key must give O = 0"
        assert np.all(np.isneginf(l64)), "a row with no visible key must give LSE = -inf"
    keep = [r for r, s_ in zip(sel, seen) if s_]
    if keep:
        idx = [i for i, s_ in enumerate(seen) if s_]
        compare(o_gpu, lse_gpu, o_ref[:, idx], lse_ref[:, :, idx], rows=keep)
