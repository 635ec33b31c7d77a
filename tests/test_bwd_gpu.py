"""Backward-pass parity: attn_bwd (through the C ABI) against the fp64
oracle's chain-rule gradients.

The forward runs on the GPU (its O and LSE feed the backward, as in use);
the oracle recomputes everything from the same rounded inputs in fp64.
Shapes: single tiles, ragged query and key tails, sq != sk, several units
per CTA, every head dim and both dtypes; the same with the causal mask,
including query tiles that see no key at all (sq > sk + 128).

Tolerance. The gradients are sums over keys (dQ) or query rows (dK, dV) of
products that go through 16-bit P and dS on the tensor core, so their error
scales with their size: max |g - g_ref| <= 2e-2 * (1 + max |g_ref|) for each
of dQ, dK, dV (the forward's 2e-2 on O, scaled by the gradient's magnitude).
"""
import math

import numpy as np
import pytest
import torch

import workloads
from parity import to_np64

pytestmark = pytest.mark.gpu


def _check_bwd(ea, oracle_mod, b, sq, sk, h, d, dtype, seed, causal=False):
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    do = torch.randn((b, sq, h, d), generator=g).to(dtype)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    scale = 1 / math.sqrt(d)
    o, lse = ea.attn_fwd(qd, kd, vd, scale=scale, causal=causal)
    dq, dk, dv = ea.attn_bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal)
    status = ea.attn_get_device_status()
    assert status == ea.ATTN_OK, f"status {status}, site {ea.attn_last_timeout_site():#x}"
    rq, rk, rv = oracle_mod.attention_backward(q, k, v, do, scale, causal=causal)
    errs = {}
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        g64 = to_np64(got)
        assert np.all(np.isfinite(g64)), f"non-finite {name}"
        err = float(np.abs(g64 - ref).max())
        bound = 2e-2 * (1.0 + float(np.abs(ref).max()))
        errs[name] = (err, bound)
        assert err <= bound, f"{name}: max err {err:.3e} > {bound:.3e} (max |ref| {np.abs(ref).max():.3e})"
    return errs


@pytest.mark.parametrize("b,sq,sk,h,d", [(1, 128, 128, 1, 128), (2, 300, 200, 3, 128),
                                         (1, 64, 1000, 2, 64), (1, 513, 257, 2, 32),
                                         (3, 100, 130, 2, 16), (1, 1, 77, 1, 128)])
def test_bwd_shapes(gpu, oracle_mod, b, sq, sk, h, d):
    _check_bwd(gpu, oracle_mod, b, sq, sk, h, d, torch.bfloat16, 91)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_bwd_fp16(gpu, oracle_mod, d):
    _check_bwd(gpu, oracle_mod, 2, 200, 333, 2, d, torch.float16, 93)


def test_bwd_many_units_per_cta(gpu, oracle_mod):
    """More tiles than SMs: every persistent CTA runs several units."""
    _check_bwd(gpu, oracle_mod, 4, 512, 512, 48, 64, torch.bfloat16, 95)


@pytest.mark.parametrize("b,sq,sk,h,d", [(1, 128, 128, 1, 128), (2, 300, 300, 3, 128),
                                         (1, 64, 1000, 2, 64), (1, 513, 257, 2, 32),
                                         (2, 300, 200, 2, 128), (3, 100, 130, 2, 16),
                                         (1, 1, 77, 1, 128), (1, 777, 777, 2, 64)])
def test_bwd_causal_shapes(gpu, oracle_mod, b, sq, sk, h, d):
    _check_bwd(gpu, oracle_mod, b, sq, sk, h, d, torch.bfloat16, 97, causal=True)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_bwd_causal_fp16(gpu, oracle_mod, d):
    _check_bwd(gpu, oracle_mod, 2, 333, 200, 2, d, torch.float16, 99, causal=True)


def test_bwd_causal_many_units_per_cta(gpu, oracle_mod):
    """Causal with more tiles than SMs: units of very different lengths."""
    _check_bwd(gpu, oracle_mod, 4, 640, 640, 48, 64, torch.bfloat16, 101, causal=True)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_graph_capture_and_user_stream_match_eager(gpu, causal):
    """The key-tile and query-tile kernels run side by side on the caller's
    stream and a library stream joined back to it; under graph capture they
    run one after the other on the captured stream. Both give bit-identical
    gradients, also when the call is made on a user stream."""
    b, s, h, d = 2, 700, 8, 128
    q, k, v = (t.cuda() for t in workloads.make_qkv(b, s, s, h, d, torch.bfloat16, seed=113))
    do = torch.randn((b, s, h, d), generator=torch.Generator().manual_seed(114)).to(
        torch.bfloat16).cuda()
    o, lse = gpu.attn_fwd(q, k, v, causal=causal)
    ref = gpu.attn_bwd(q, k, v, o, lse, do, causal=causal)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        got = gpu.attn_bwd(q, k, v, o, lse, do, causal=causal)
    side.synchronize()
    for a_, b_ in zip(ref, got):
        assert torch.equal(a_, b_)
    outs = [torch.empty_like(t) for t in ref]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gpu.attn_bwd(q, k, v, o, lse, do, dq=outs[0], dk=outs[1], dv=outs[2], causal=causal)
    graph.replay()
    torch.cuda.synchronize()
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    for a_, b_ in zip(ref, outs):
        assert torch.equal(a_, b_)
