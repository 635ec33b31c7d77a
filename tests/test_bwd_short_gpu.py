"""Parity of the short backward kernel (one (batch, head) per work item, all
of its keys in one row of S: d 16 or 32, at most 256 query rows and 160
keys, not causal) against the fp64 oracle's chain-rule gradients, through
the C ABI. attn_bwd takes it for those shapes; the debug flag
ATTN_DEBUG_GENERAL_BWD sends the same calls to the key-tile and query-tile
kernels, which must agree with the oracle too.

Shapes (80 (batch, head) items, or one tile on each side, so that the short
kernel is the one that runs): key counts on both sides of every 16- and
32-key chunk edge and of the 128-key M tile (1, 5, 31, 32, 33, 64, 100, 128,
129, 150, 160), query counts from one row to two ragged 128-row tiles (1, 2,
127, 128, 129, 200, 256),
both head dims and dtypes, the flash-attn timing issue's small-head shapes
(b2 s50 and, with fewer batches, s150 at h16 d16), far more items than SMs,
large scores, and a timeout that the context survives.
Tolerance as in the other backward tests: max |g - g_ref| <= 2e-2 (1 + max
|g_ref|) for each of dQ, dK, dV.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from parity import to_np64

pytestmark = pytest.mark.gpu

# attn_bwd takes the short kernel for these shapes when there are at least
# half as many (batch, head) items as SMs (or one tile on each side): 40
# batches of 2 heads are 80 items, past half of this part's 152 SMs
ITEMS_B = 40


def _grads(ea, q, k, v, do, scale, general=False):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = ea.attn_fwd(qd, kd, vd, scale=scale)
    if general:
        ea.attn_debug_set_flags(ea.ATTN_DEBUG_GENERAL_BWD)
    try:
        out = ea.attn_bwd(qd, kd, vd, o, lse, dod, scale=scale)
    finally:
        ea.attn_debug_set_flags(0)
    status = ea.attn_get_device_status()
    assert status == ea.ATTN_OK, f"status {status}, site {ea.attn_last_timeout_site():#x}"
    return out


def _check(ea, oracle_mod, b, sq, sk, h, d, dtype, seed, q_mul=1.0, general=False):
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=seed)
    if q_mul != 1.0:
        q = (q.float() * q_mul).to(dtype)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn((b, sq, h, d), generator=g).to(dtype)
    scale = 1 / math.sqrt(d)
    got = _grads(ea, q, k, v, do, scale, general)
    ref = oracle_mod.attention_backward(q, k, v, do, scale)
    for name, gt, rf in zip(("dq", "dk", "dv"), got, ref):
        g64 = to_np64(gt)
        assert np.all(np.isfinite(g64)), f"non-finite {name}"
        err = float(np.abs(g64 - rf).max())
        bound = 2e-2 * (1.0 + float(np.abs(rf).max()))
        assert err <= bound, f"{name}: max err {err:.3e} > {bound:.3e}"
    return got


@pytest.mark.parametrize("sk", [1, 5, 31, 32, 33, 64, 100, 128, 129, 150, 160])
@pytest.mark.parametrize("d", [16, 32])
def test_key_counts_and_head_dims(gpu, oracle_mod, sk, d):
    dtype = torch.float16 if d == 16 else torch.bfloat16
    _check(gpu, oracle_mod, ITEMS_B, 150, sk, 2, d, dtype, seed=401 + sk)


@pytest.mark.parametrize("sq", [1, 2, 127, 128, 129, 200, 256])
def test_query_counts(gpu, oracle_mod, sq):
    _check(gpu, oracle_mod, ITEMS_B, sq, 150, 2, 16, torch.float16, seed=421 + sq)


@pytest.mark.parametrize("d", [16, 32])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_dtypes(gpu, oracle_mod, d, dtype):
    _check(gpu, oracle_mod, ITEMS_B, 140, 120, 2, d, dtype, seed=431 + d)


@pytest.mark.parametrize("b,s", [(2, 50), (64, 150)])
def test_timing_issue_shapes_both_kernels(gpu, oracle_mod, b, s):
    """h16 d16 fp16 at s = 50 (b2, the issue's own shape) and s = 150 (b64:
    1024 items, several per CTA; the issue's b512 is the bench shape): the
    short kernel and the tile kernels each match the oracle, and each other."""
    g1 = _check(gpu, oracle_mod, b, s, s, 16, 16, torch.float16, seed=441 + s)
    g2 = _check(gpu, oracle_mod, b, s, s, 16, 16, torch.float16, seed=441 + s, general=True)
    for a_, b_ in zip(g1, g2):
        ref = max(float(a_.float().abs().max()), 1.0)
        assert (a_.float() - b_.float()).abs().max().item() <= 2e-2 * ref


def test_large_scores(gpu, oracle_mod):
    """Scores spread over tens of units: P is exp(S - LSE) with the
    forward's LSE, so nothing overflows however far apart the scores are."""
    _check(gpu, oracle_mod, ITEMS_B, 130, 150, 2, 32, torch.bfloat16, seed=451, q_mul=6.0)


def test_repeat_calls_are_deterministic(gpu):
    q, k, v = (t.cuda() for t in workloads.make_qkv(10, 150, 150, 8, 16, torch.float16, seed=461))
    do = torch.randn((10, 150, 8, 16), generator=torch.Generator().manual_seed(462)).to(
        torch.float16).cuda()
    o, lse = gpu.attn_fwd(q, k, v)
    a1 = gpu.attn_bwd(q, k, v, o, lse, do)
    a2 = gpu.attn_bwd(q, k, v, o, lse, do)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    for x, y in zip(a1, a2):
        assert torch.equal(x, y)


def test_graph_capture_and_user_stream_match_eager(gpu):
    """The short kernel (and the D = rowsum(dO * O) kernel before it) on a
    user stream and inside a captured graph give bit-identical gradients."""
    q, k, v = (t.cuda() for t in workloads.make_qkv(10, 150, 150, 8, 16, torch.float16, seed=481))
    do = torch.randn((10, 150, 8, 16), generator=torch.Generator().manual_seed(482)).to(
        torch.float16).cuda()
    o, lse = gpu.attn_fwd(q, k, v)
    ref = gpu.attn_bwd(q, k, v, o, lse, do)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        got = gpu.attn_bwd(q, k, v, o, lse, do)
    side.synchronize()
    for a_, b_ in zip(ref, got):
        assert torch.equal(a_, b_)
    outs = [torch.empty_like(t) for t in ref]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gpu.attn_bwd(q, k, v, o, lse, do, dq=outs[0], dk=outs[1], dv=outs[2])
    graph.replay()
    torch.cuda.synchronize()
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    for a_, b_ in zip(ref, outs):
        assert torch.equal(a_, b_)


def test_timeout_and_recovery(gpu):
    """ATTN_DEBUG_SKIP_LOADS: the producer issues nothing, the MMA issuer's
    wait for the first item's inputs runs out after its bound, the kernel
    returns, the status reports it, and the next call works."""
    q, k, v = (t.cuda() for t in workloads.make_qkv(1, 100, 100, 2, 16, torch.float16, seed=471))
    do = torch.randn((1, 100, 2, 16), generator=torch.Generator().manual_seed(472)).to(
        torch.float16).cuda()
    o, lse = gpu.attn_fwd(q, k, v)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    gpu.attn_debug_set_flags(gpu.ATTN_DEBUG_SKIP_LOADS)
    try:
        gpu.attn_bwd(q, k, v, o, lse, do)
    finally:
        gpu.attn_debug_set_flags(0)
    assert gpu.attn_get_device_status() == gpu.ATTN_ERR_DEVICE_TIMEOUT
    assert gpu.attn_last_timeout_site() >> 8 == 3
    dq, dk, dv = gpu.attn_bwd(q, k, v, o, lse, do)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    assert all(torch.isfinite(t.float()).all() for t in (dq, dk, dv))
