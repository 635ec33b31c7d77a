"""Split-KV decode parity: the CUDA path (through the C ABI) against the fp64 oracle.

Shapes: the two decode problems of the flash-decoding issue (b8 h48 sk8192,
where the heuristic must not split, and b1 h16 sk32768 with num_splits in
{0, 2, 4, 8, 16}), plus the split/combine edge cases: more splits than key
blocks, empty splits, a key count that is not a multiple of the block,
every head dim and fp16 through the explicit-dtype entry point. Several
query rows (the issue's 1 to 10 new tokens, and more) run on the
tensor-core kernel split along the keys; they get the same cases.
Tolerance: max |O - O_ref| <= 2e-2, max |LSE - LSE_ref| <= 1e-3.
"""
import math

import pytest
import torch

import workloads
from parity import compare, to_np64

pytestmark = pytest.mark.gpu


def run_decode(ea, q, k, v, scale, splits):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = ea.attn_decode_splitkv(qd, kd, vd, scale=scale, num_splits=splits)
    assert ea.attn_get_device_status() == ea.ATTN_OK
    return o, lse


@pytest.fixture(scope="module")
def case_b(oracle_mod):
    w = workloads.WORKLOADS["decode_b1_h16_sk32768"]
    q, k, v = workloads.make_workload(w)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, w.scale)
    return w, (q, k, v), (o_ref, lse_ref)


@pytest.mark.parametrize("splits", [0, 1, 2, 4, 8, 16])
def test_case_b_splits(gpu, case_b, splits):
    w, (q, k, v), (o_ref, lse_ref) = case_b
    o, lse = run_decode(gpu, q, k, v, w.scale, splits)
    compare(o, lse, o_ref, lse_ref)


def test_case_b_heuristic_splits(gpu):
    w = workloads.WORKLOADS["decode_b1_h16_sk32768"]
    s = gpu.attn_decode_num_splits(w.b, w.sq, w.sk, w.h, w.d)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert s > 1 and w.b * w.h * s <= sms < w.b * w.h * (s + 1)


def test_case_a_heuristic_and_parity(gpu, oracle_mod):
    w = workloads.WORKLOADS["decode_b8_h48_sk8192"]
    assert gpu.attn_decode_num_splits(w.b, w.sq, w.sk, w.h, w.d) == 1
    q, k, v = workloads.make_workload(w)
    o, lse = run_decode(gpu, q, k, v, w.scale, 0)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, w.scale)
    compare(o, lse, o_ref, lse_ref)


def test_split_equals_unsplit(gpu, case_b):
    w, (q, k, v), _ = case_b
    o1, l1 = run_decode(gpu, q, k, v, w.scale, 1)
    for s in (3, 7, 64):
        o2, l2 = run_decode(gpu, q, k, v, w.scale, s)
        assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
        assert (l1 - l2).abs().max().item() <= 1e-4


@pytest.mark.parametrize("sk,splits", [
    (310, 4),     # 5 key blocks over 4 splits of 2 blocks: the last split is empty
    (64, 8),      # one block, more splits asked than blocks
    (1, 3),       # a single key
    (1000, 1000),  # clamped to the block count
    (4097, 5),    # a one-row tail block
])
def test_split_edges(gpu, oracle_mod, sk, splits):
    b, sq, h, d = 2, 1, 3, 128
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=17)
    o, lse = run_decode(gpu, q, k, v, 1 / math.sqrt(d), splits)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(d))
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("sq", [2, 3, 5, 10])
def test_several_query_rows(gpu, oracle_mod, sq):
    b, sk, h, d = 2, 3000, 6, 128
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=19)
    for splits in (0, 1, 6):
        o, lse = run_decode(gpu, q, k, v, 1 / math.sqrt(d), splits)
        o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(d))
        compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_head_dims_and_dtypes(gpu, oracle_mod, d, dtype):
    b, sq, sk, h = 2, 1, 5000, 4
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=23)
    for splits in (0, 1, 5):
        o, lse = run_decode(gpu, q, k, v, 1 / math.sqrt(d), splits)
        o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(d))
        compare(o, lse, o_ref, lse_ref)


def test_decode_matches_forward(gpu):
    b, sq, sk, h, d = 1, 1, 9000, 8, 128
    q, k, v = (t.cuda() for t in workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=29))
    o1, l1 = gpu.attn_fwd(q, k, v)
    o2, l2 = gpu.attn_decode_splitkv(q, k, v, num_splits=0)
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-4


def test_bf16_entry_point_through_raw_abi(gpu, oracle_mod):
    """attn_decode_splitkv (no dtype argument) is the bf16 entry point."""
    import ctypes

    b, sq, sk, h, d = 1, 1, 700, 2, 128
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=31)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty(b, h, sq, dtype=torch.float32, device="cuda")
    lib = gpu.load_library()
    rc = lib.attn_decode_splitkv(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(),
                                 lse.data_ptr(), b, sq, sk, h, d, 1 / math.sqrt(d), 3,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(d))
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("sq", [2, 7, 10, 16, 130, 300])
@pytest.mark.parametrize("splits", [0, 1, 3, 64])
def test_many_rows_split_on_tensor_cores(gpu, oracle_mod, sq, splits):
    """Several query rows share each K/V read: the key range is split into
    whole 128-key tiles (3 or 64 asked; 64 exceeds the 24 tiles of sk = 3000
    and is clamped), partials reduced by the combine kernel. sk = 3000 leaves
    a ragged last tile; sq = 130 and 300 span two query tiles and a ragged
    second unit."""
    b, sk, h, d = 2, 3000, 3, 128
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=43)
    o, lse = run_decode(gpu, q, k, v, 1 / math.sqrt(d), splits)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(d))
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_many_rows_head_dims_and_dtypes(gpu, oracle_mod, d, dtype):
    b, sq, sk, h = 1, 5, 1000, 4
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=47)
    for splits in (0, 1, 4):
        o, lse = run_decode(gpu, q, k, v, 1 / math.sqrt(d), splits)
        o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(d))
        compare(o, lse, o_ref, lse_ref)


def test_many_rows_split_equals_unsplit_and_forward(gpu):
    b, sq, sk, h, d = 1, 10, 20000, 6, 128
    q, k, v = (t.cuda() for t in workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=53))
    o0, l0 = gpu.attn_fwd(q, k, v)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    for s in (0, 1, 2, 9, 157):
        o1, l1 = gpu.attn_decode_splitkv(q, k, v, num_splits=s)
        assert gpu.attn_get_device_status() == gpu.ATTN_OK
        assert (o0.float() - o1.float()).abs().max().item() <= 1e-2
        assert (l0 - l1).abs().max().item() <= 1e-4


def test_issue_workload_few_new_rows(gpu, oracle_mod):
    """The issue's decode: batch 8, 48 heads, 1 to 10 new query rows (here
    sk = 512 to keep the oracle quick): one split, every row checked."""
    b, sk, h, d = 8, 512, 48, 128
    for sq in (1, 2, 10):
        assert gpu.attn_decode_num_splits(b, sq, 8192, h, d) == 1
        q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=59)
        o, lse = run_decode(gpu, q, k, v, 1 / math.sqrt(d), 0)
        o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(d))
        compare(o, lse, o_ref, lse_ref)
