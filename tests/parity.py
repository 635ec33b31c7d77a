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
