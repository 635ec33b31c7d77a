"""The split decode's reduce inside the split kernel (the split of a
(batch, head) that finishes last reduces it, found through per-stream
arrival counters), against the fp64 oracle.

Cases: many calls in a row on one stream with changing split counts and
shapes (the counters must come back to zero after every call), a shape
with more (batch, head) pairs than the first counter array holds (it is
grown), partials that outgrow the stream's workspace, a second stream with
its own counters, results bit-identical to
the separate reduce kernel, which a call captured into a CUDA graph uses
(replayed twice), and the paged cache. Tolerance: |O| 2e-2, LSE 1e-3.
"""
import math

import pytest
import torch

import workloads
from parity import compare

pytestmark = pytest.mark.gpu


def _qkv(b, sk, h, d=128, seed=5):
    return workloads.make_qkv(b, 1, sk, h, d, torch.bfloat16, seed=seed)


def test_counters_return_to_zero_across_calls(gpu, oracle_mod):
    cases = [(1, 5000, 4, 7), (2, 3000, 8, 3), (1, 5000, 4, 2), (3, 777, 5, 9), (1, 5000, 4, 7),
             (2, 3000, 8, 16), (3, 777, 5, 4)]
    data = {}
    for b, sk, h, splits in cases:
        if (b, sk, h) not in data:
            q, k, v = _qkv(b, sk, h, seed=b * 100 + h)
            data[(b, sk, h)] = ((q, k, v), oracle_mod.attention(q, k, v, 1 / math.sqrt(128)),
                                tuple(t.cuda() for t in (q, k, v)))
        _, (o_ref, lse_ref), (qd, kd, vd) = data[(b, sk, h)]
        o, lse = gpu.attn_decode_splitkv(qd, kd, vd, num_splits=splits)
        assert gpu.attn_get_device_status() == gpu.ATTN_OK
        compare(o, lse, o_ref, lse_ref)


def test_counter_array_grows(gpu, oracle_mod):
    # 6 x 200 = 1200 (batch, head) pairs: more than the first array's 1024
    q, k, v = _qkv(6, 600, 200, d=64, seed=11)
    o, lse = gpu.attn_decode_splitkv(q.cuda(), k.cuda(), v.cuda(), num_splits=3)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    compare(o, lse, *oracle_mod.attention(q, k, v, 1 / math.sqrt(64)))


def test_second_stream_and_bit_identity_with_reduce_kernel(gpu, oracle_mod):
    q, k, v = _qkv(2, 4100, 6, seed=13)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(128))
    o1, l1 = gpu.attn_decode_splitkv(qd, kd, vd, num_splits=5)
    s2 = torch.cuda.Stream()
    with torch.cuda.stream(s2):
        o2, l2 = gpu.attn_decode_splitkv(qd, kd, vd, num_splits=5)
    s2.synchronize()
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    compare(o1, l1, o_ref, lse_ref)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # a captured call reduces with the second kernel; same bits
    o3 = torch.empty_like(o1)
    l3 = torch.empty_like(l1)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            gpu.attn_decode_splitkv(qd, kd, vd, num_splits=5, out=o3, lse=l3)
    for _ in range(2):
        o3.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert gpu.attn_get_device_status() == gpu.ATTN_OK
        assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_paged_in_kernel_reduce(gpu, oracle_mod):
    b, h, d, page = 3, 4, 128, 256
    lens = [1000, 3, 2048]
    npages = [math.ceil(n / page) for n in lens]
    total = sum(npages) + 2
    g = torch.Generator().manual_seed(17)
    kp = torch.randn((total, page, h, d), generator=g).bfloat16()
    vp = torch.randn((total, page, h, d), generator=g).bfloat16()
    q = torch.randn((b, 1, h, d), generator=g).bfloat16()
    perm = torch.randperm(total, generator=g)
    table = torch.zeros((b, max(npages)), dtype=torch.int32)
    pos = 0
    for i, n in enumerate(npages):
        table[i, :n] = perm[pos:pos + n].to(torch.int32)
        pos += n
    seqlens = torch.tensor(lens, dtype=torch.int32)
    for splits in (4, 2, 4):
        o, lse = gpu.attn_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), seqlens.cuda(),
                                       num_splits=splits)
        assert gpu.attn_get_device_status() == gpu.ATTN_OK
        o_ref, lse_ref = oracle_mod.paged_attention(q, kp, vp, table, seqlens, 1 / math.sqrt(d))
        compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("splits", [16, 17, 40, 100])
def test_many_splits(gpu, oracle_mod, splits):
    """Up to 16 splits are reduced from registers in one pass; more take the
    looped form (in the split kernel and in the reduce kernel, sq > 1)."""
    for sq in (1, 3):
        q, k, v = workloads.make_qkv(2, sq, 20000, 3, 128, torch.bfloat16, seed=splits + sq)
        o, lse = gpu.attn_decode_splitkv(q.cuda(), k.cuda(), v.cuda(), num_splits=splits)
        assert gpu.attn_get_device_status() == gpu.ATTN_OK
        compare(o, lse, *oracle_mod.attention(q, k, v, 1 / math.sqrt(128)))


def test_stream_workspace_grows_and_is_reused(gpu, oracle_mod):
    """Partials of 16 splits x 384 (batch, head) rows x d = 128 in fp32 (3 MB)
    outgrow the stream's first workspace; smaller calls after it reuse the
    grown one."""
    big = _qkv(8, 4096, 48, seed=21)
    small = _qkv(1, 3000, 4, seed=22)
    refs = {id(x): oracle_mod.attention(*x, 1 / math.sqrt(128)) for x in (big, small)}
    for x, splits in ((small, 5), (big, 16), (small, 7), (big, 9), (small, 3)):
        o, lse = gpu.attn_decode_splitkv(*(t.cuda() for t in x), num_splits=splits)
        assert gpu.attn_get_device_status() == gpu.ATTN_OK
        compare(o, lse, *refs[id(x)])


def test_release_then_decode_again(gpu, oracle_mod):
    """attn_release_workspace frees the per-stream counters and partials; the
    next split decode on the same stream makes them again."""
    q, k, v = _qkv(1, 5000, 4, seed=23)
    ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(128))
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    for _ in range(2):
        o, lse = gpu.attn_decode_splitkv(qd, kd, vd, num_splits=6)
        assert gpu.attn_get_device_status() == gpu.ATTN_OK
        compare(o, lse, *ref)
        gpu.attn_release_workspace()


def test_several_rows_share_the_stream_workspace(gpu, oracle_mod):
    """Several-row decodes (tensor-core kernel, partials in the stream's
    workspace, reduce kernel) interleaved with one-row decodes (in-kernel
    reduce) on one stream, with growing and shrinking partials; then the same
    several-row call captured into a graph (per-call workspace) gives the
    same bits."""
    cases = [(1, 1, 5000, 4, 7), (2, 10, 3000, 8, 3), (1, 1, 5000, 4, 9), (1, 16, 9000, 6, 40),
             (2, 10, 3000, 8, 3), (1, 2, 700, 3, 5)]
    inputs = {c: workloads.make_qkv(c[0], c[1], c[2], c[3], 128, torch.bfloat16, seed=31 + i)
              for i, c in enumerate(cases)}
    refs = {c: oracle_mod.attention(*inputs[c], 1 / math.sqrt(128)) for c in cases}
    outs = {}
    for c in cases:
        o, lse = gpu.attn_decode_splitkv(*(t.cuda() for t in inputs[c]), num_splits=c[4])
        assert gpu.attn_get_device_status() == gpu.ATTN_OK
        compare(o, lse, *refs[c])
        outs[c] = (o, lse)
    c = cases[1]
    qd, kd, vd = (t.cuda() for t in inputs[c])
    o3 = torch.empty_like(outs[c][0])
    l3 = torch.empty_like(outs[c][1])
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            gpu.attn_decode_splitkv(qd, kd, vd, num_splits=c[4], out=o3, lse=l3)
    graph.replay()
    torch.cuda.synchronize()
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    assert torch.equal(outs[c][0], o3) and torch.equal(outs[c][1], l3)
