"""Bounded waits: a kernel whose loads never arrive returns with a timeout
status instead of hanging, and the CUDA context stays usable afterwards.

The failure is made on the host: the debug flag ATTN_DEBUG_SKIP_LOADS makes
the TMA producer issue nothing, so no copy is ever in flight and every wait
on a "full" barrier runs out after its bound (about two seconds). No fault,
trap or unbounded loop is involved.
"""
import time

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def _inputs(sq, sk):
    return [t.cuda() for t in workloads.make_qkv(1, sq, sk, 2, 128, torch.bfloat16, seed=37)]


@pytest.mark.parametrize("which", ["fwd", "fwd_two_tiles", "decode", "decode_rows"])
def test_skipped_loads_time_out_and_recover(gpu, which):
    # fwd: 64 rows (the one-tile forward kernel); fwd_two_tiles: 300 rows
    # (the two-tile kernel); decode: one row (the CUDA-core split kernel);
    # decode_rows: 10 rows (the one-tile forward kernel on key ranges)
    sq = {"fwd": 64, "fwd_two_tiles": 300, "decode": 1, "decode_rows": 10}[which]
    q, k, v = _inputs(sq, 256)
    call = (lambda: gpu.attn_fwd(q, k, v)) if which.startswith("fwd") else (
        lambda: gpu.attn_decode_splitkv(q, k, v, num_splits=2))
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    gpu.attn_debug_set_flags(gpu.ATTN_DEBUG_SKIP_LOADS)
    try:
        call()
    finally:
        gpu.attn_debug_set_flags(0)
    t0 = time.time()
    status = gpu.attn_get_device_status()
    elapsed = time.time() - t0
    assert status == gpu.ATTN_ERR_DEVICE_TIMEOUT
    assert elapsed < 60
    kernel = gpu.attn_last_timeout_site() >> 8
    assert kernel == (2 if which == "decode" else 1)
    # the status word was cleared and the context still works
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    o, lse = call()
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
