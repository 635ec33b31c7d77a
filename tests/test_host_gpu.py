"""Host-buffer forward (attn_fwd_host through the C ABI): the copy /
compute / copy-back pipeline gives, for every chunking it uses, the same
bits as attn_fwd on device copies of the inputs, and matches the fp64
oracle within the forward's tolerance (|O| 2e-2, LSE 1e-3).

Chunkings covered: several batches (one and more per chunk, more batches
than chunks), one non-causal batch cut into query-row ranges (ragged last
range, LSE gathered back into [h, sq]), causal batches (whole batches),
pinned and pageable host memory, fp16 and bf16, and the call queued
without synchronising (sync=False) and read after the stream is done.
"""
import math

import pytest
import torch

import workloads
from parity import compare_masked

pytestmark = pytest.mark.gpu


def _pinned(t, pin):
    return t.pin_memory() if pin else t.clone()


def _check(ea, oracle_mod, b, sq, sk, h, d, dtype, causal=False, pin=True, seed=71, sync=True):
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=seed)
    scale = 1.0 / math.sqrt(d)
    hq, hk, hv = (_pinned(t, pin) for t in (q, k, v))
    if pin:
        o, lse = ea.attn_fwd_host(hq, hk, hv, scale=scale, causal=causal, sync=sync)
    else:
        o = torch.empty_like(q)
        lse = torch.empty((b, h, sq), dtype=torch.float32)
        ea.attn_fwd_host(hq, hk, hv, scale=scale, out=o, lse=lse, causal=causal, sync=sync)
    if not sync:
        torch.cuda.current_stream().synchronize()
    assert ea.attn_get_device_status() == ea.ATTN_OK
    assert o.device.type == "cpu" and lse.device.type == "cpu"
    # bit-identical to the device-pointer call
    od, ld = ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal)
    assert torch.equal(o, od.cpu()), "O differs from attn_fwd"
    assert torch.equal(lse, ld.cpu()), "LSE differs from attn_fwd"
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale, causal=causal)
    compare_masked(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("b,sq,sk,h,d", [(4, 300, 200, 2, 128), (2, 64, 1000, 3, 64),
                                         (11, 130, 77, 2, 32), (3, 1, 513, 2, 128),
                                         (4, 512, 512, 3, 128), (3, 1000, 333, 2, 64),
                                         (9, 600, 100, 2, 32)])
def test_host_batches(gpu, oracle_mod, b, sq, sk, h, d):
    _check(gpu, oracle_mod, b, sq, sk, h, d, torch.bfloat16)


@pytest.mark.parametrize("sq,sk", [(512, 300), (1000, 777), (1300, 1300)])
def test_host_one_batch_by_rows(gpu, oracle_mod, sq, sk):
    _check(gpu, oracle_mod, 1, sq, sk, 3, 128, torch.bfloat16)


@pytest.mark.parametrize("b", [1, 3])
def test_host_causal(gpu, oracle_mod, b):
    _check(gpu, oracle_mod, b, 700, 500, 2, 64, torch.bfloat16, causal=True)


def test_host_fp16_pageable(gpu, oracle_mod):
    _check(gpu, oracle_mod, 2, 600, 333, 2, 16, torch.float16, pin=False)


def test_host_queued_then_synchronised(gpu, oracle_mod):
    _check(gpu, oracle_mod, 4, 512, 512, 4, 128, torch.bfloat16, sync=False)


def test_host_rejects_device_tensors(gpu):
    q = torch.zeros((1, 8, 1, 16), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        gpu.attn_fwd_host(q, q, q)


def test_host_refuses_graph_capture(gpu):
    """The pipeline uses the library's own copy streams: a captured call is
    refused (ATTN_ERR_UNSUPPORTED) and the capture itself stays intact."""
    q = torch.zeros((1, 8, 1, 16), dtype=torch.float16).pin_memory()
    o = torch.empty_like(q).pin_memory()
    lse = torch.empty((1, 1, 8), dtype=torch.float32).pin_memory()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    x = torch.zeros(4, device="cuda")
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            x.add_(1)
            with pytest.raises(gpu.AttnError) as err:
                gpu.attn_fwd_host(q, q, q, out=o, lse=lse, sync=False)
            assert err.value.status == gpu.ATTN_ERR_UNSUPPORTED
    graph.replay()
    torch.cuda.synchronize()
    assert x.tolist() == [1.0] * 4
