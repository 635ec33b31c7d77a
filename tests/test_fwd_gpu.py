"""Forward parity: the CUDA path (through the C ABI) against the fp64 oracle.

Shapes: the tiny and small-head problems of the flash-attn timing issue
(head dim 16, fp16), the b4 s512 h32 d128 bf16 problem of "Why
FlashAttention is fast" on every row, a problem with more units than SMs on
every row, the long b1 s8192 h32 d128 problem on 256 sampled rows, and edge
cases: ragged query/key tails, fewer keys than one tile, single rows and
keys, every head dim, both dtypes, zero and negative scale.
Tolerance: max |O - O_ref| <= 2e-2 and max |LSE - LSE_ref| <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from parity import compare

pytestmark = pytest.mark.gpu


def run_fwd(ea, q, k, v, scale):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = ea.attn_fwd(qd, kd, vd, scale=scale)
    assert ea.attn_get_device_status() == ea.ATTN_OK
    return o, lse


def check_full(ea, oracle_mod, b, sq, sk, h, d, dtype, scale=None, seed=42):
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=seed)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o, lse = run_fwd(ea, q, k, v, scale)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale)
    return compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("name", ["tiny_fwd", "small_head_b2_s50", "small_head_b2_s300",
                                  "small_head_b512_s150"])
def test_pages_small_shapes_all_rows(gpu, oracle_mod, name):
    w = workloads.WORKLOADS[name]
    check_full(gpu, oracle_mod, w.b, w.sq, w.sk, w.h, w.d, w.dtype)


def test_mid_fwd_all_rows(gpu, oracle_mod):
    """The b4 s512 h32 d128 bf16 problem of "Why FlashAttention is fast",
    every query row of every (batch, head) against the oracle."""
    w = workloads.WORKLOADS["mid_fwd"]
    q, k, v = workloads.make_workload(w)
    o, lse = run_fwd(gpu, q, k, v, w.scale)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, w.scale)
    compare(o, lse, o_ref, lse_ref)


def test_several_units_per_cta_all_rows(gpu, oracle_mod):
    """More 256-row units than SMs (b2 s1024 h48 d128: 384 units), so every
    persistent CTA runs several units and reuses its Q buffer and O
    accumulator; every row is compared."""
    b, s, h, d = 2, 1024, 48, 128
    q, k, v = workloads.make_qkv(b, s, s, h, d, torch.bfloat16, seed=29)
    scale = 1 / math.sqrt(d)
    o, lse = run_fwd(gpu, q, k, v, scale)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale)
    compare(o, lse, o_ref, lse_ref)


def test_long_fwd_strided_rows(gpu, oracle_mod):
    w = workloads.WORKLOADS["long_fwd"]
    q, k, v = workloads.make_workload(w)
    o, lse = run_fwd(gpu, q, k, v, w.scale)
    rows = workloads.LONG_FWD_ROWS
    o_ref, lse_ref = oracle_mod.attention(q, k, v, w.scale, rows=rows)
    compare(o, lse, o_ref, lse_ref, rows=rows)
    # Properties that hold for every row at any size:
    #   Jensen:          LSE >= ln sk + mean_j s_j = ln sk + scale * q . mean_j k_j
    #   Cauchy-Schwarz:  LSE <= ln sk + max_j s_j <= ln sk + scale * |q| * max_j |k_j|
    qd = q.cuda().float()
    kd = k.cuda().float()
    kmean = kd.mean(dim=1)                                   # [b, h, d]
    lower = math.log(w.sk) + w.scale * torch.einsum("bshd,bhd->bhs", qd, kmean)
    kmax = kd.norm(dim=-1).amax(dim=1)                       # [b, h]
    upper = math.log(w.sk) + w.scale * qd.norm(dim=-1).transpose(1, 2) * kmax[..., None]
    assert bool(torch.all(lse >= lower - 1e-3)), "LSE below the Jensen bound"
    assert bool(torch.all(lse <= upper + 1e-3)), "LSE above the Cauchy-Schwarz bound"


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_head_dims_and_dtypes(gpu, oracle_mod, d, dtype):
    check_full(gpu, oracle_mod, 2, 200, 333, 3, d, dtype, seed=7)


@pytest.mark.parametrize("b,sq,sk,h,d", [
    (1, 1, 1, 1, 64),        # one query, one key
    (1, 1, 5, 2, 128),       # fewer keys than a tile
    (2, 3, 128, 1, 128),     # exactly one key tile
    (1, 129, 129, 2, 64),    # one past a tile on both sides
    (1, 256, 256, 1, 128),   # both query tiles of one CTA full
    (1, 257, 300, 1, 128),   # a second CTA with one row
    (3, 700, 1000, 2, 32),   # several CTAs, ragged tails
    (1, 64, 4096, 4, 128),   # many key tiles
])
def test_edge_shapes(gpu, oracle_mod, b, sq, sk, h, d):
    check_full(gpu, oracle_mod, b, sq, sk, h, d, torch.bfloat16, seed=11)


@pytest.mark.parametrize("scale", [0.0, -0.3, 0.5])
def test_scales(gpu, oracle_mod, scale):
    check_full(gpu, oracle_mod, 1, 100, 200, 2, 64, torch.float16, scale=scale, seed=3)


def test_large_scores_stay_stable(gpu, oracle_mod):
    """Scores spanning hundreds of units exercise the running-max rescale."""
    b, sq, sk, h, d = 1, 130, 520, 2, 64
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=5)
    q = (q.float() * 6).to(torch.bfloat16)
    o, lse = run_fwd(gpu, q, k, v, 1.0)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 1.0)
    compare(o, lse, o_ref, lse_ref)


def test_increasing_scores_force_every_rescale(gpu, oracle_mod):
    """Keys whose scores grow tile after tile move the reference max on
    every tile, so every correction step runs."""
    b, sq, sk, h, d = 1, 128, 1024, 1, 64
    q = torch.ones(b, sq, h, d).to(torch.bfloat16)
    ramp = torch.linspace(0, 4, sk).view(1, sk, 1, 1)
    k = (ramp * torch.ones(b, sk, h, d)).to(torch.bfloat16)
    _, _, v = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=9)
    o, lse = run_fwd(gpu, q, k, v, 0.5)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 0.5)
    compare(o, lse, o_ref, lse_ref)


def test_equal_v_rows_give_that_row(gpu):
    b, sq, sk, h, d = 2, 150, 300, 2, 128
    q, k, _ = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=13)
    c = torch.randn(b, 1, h, d).to(torch.bfloat16)
    v = c.expand(b, sk, h, d).contiguous()
    o, _ = run_fwd(gpu, q, k, v, 1 / math.sqrt(d))
    err = (o.float().cpu() - c.float().expand(b, sq, h, d)).abs().max().item()
    assert err <= 1e-2


def test_repeat_calls_are_deterministic(gpu):
    q, k, v = (t.cuda() for t in workloads.make_qkv(2, 300, 300, 4, 64, torch.float16, seed=1))
    o1, l1 = gpu.attn_fwd(q, k, v)
    o2, l2 = gpu.attn_fwd(q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_runs_on_a_side_stream(gpu, oracle_mod):
    q, k, v = workloads.make_qkv(1, 100, 100, 2, 64, torch.bfloat16, seed=2)
    s = torch.cuda.Stream()
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        o, lse = gpu.attn_fwd(qd, kd, vd)
    s.synchronize()
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / 8)
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_output_only_16_byte_aligned(gpu, oracle_mod, d):
    """O at an address that is 16- but not 32-byte aligned (the ABI's
    minimum) takes the 16-byte store path and gives the same result."""
    b, sq, sk, h = 1, 200, 300, 3
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=41)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    n = q.numel()
    buf = torch.empty(n + 16, dtype=torch.bfloat16, device="cuda")
    base = buf.data_ptr()
    off = next(e for e in range(16) if (base + 2 * e) % 32 == 16)
    out = buf[off:off + n].view(q.shape)
    assert out.data_ptr() % 16 == 0 and out.data_ptr() % 32 != 0
    o, lse = gpu.attn_fwd(qd, kd, vd, out=out)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(d))
    compare(out, lse, o_ref, lse_ref)
