"""Parity of the short forward kernel (every key of a head in one tile: at
most 256 keys, head dims 16, 32 and 64) against the fp64 oracle, through
the C ABI. attn_fwd takes it for those shapes; the debug flag
ATTN_DEBUG_GENERAL_FWD sends the same calls to the general key-tile-loop
kernel, which must agree with the oracle too.

Shapes: key counts on both sides of every 32-column chunk edge and of the
slot widths (1, 5, 31, 32, 33, 100, 128, 150, 160, 161, 192, 224, 255, 256),
query counts from one row to several ragged 128-row tiles, grouped items
(head dim 16, heads in fours: 32-row query blocks of four heads), every head dim,
both dtypes, zero and negative scale, and far more tiles than SMs so that
every TMEM slot and shared-memory stage is reused many times. Tolerance as
everywhere: max |O - O_ref| <= 2e-2, max |LSE - LSE_ref| <= 1e-3.
"""
import math

import pytest
import torch

import workloads
from parity import compare

pytestmark = pytest.mark.gpu


def _run(ea, q, k, v, scale, general=False):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    if general:
        ea.attn_debug_set_flags(ea.ATTN_DEBUG_GENERAL_FWD)
    try:
        o, lse = ea.attn_fwd(qd, kd, vd, scale=scale)
    finally:
        ea.attn_debug_set_flags(0)
    assert ea.attn_get_device_status() == ea.ATTN_OK
    return o, lse


@pytest.mark.parametrize("sk", [1, 5, 31, 32, 33, 100, 128, 150, 160, 161, 192, 224, 255, 256])
@pytest.mark.parametrize("d", [16, 32, 64])
def test_key_counts_and_head_dims(gpu, oracle_mod, sk, d):
    b, sq, h = 2, 150, 3
    dtype = torch.float16 if d == 16 else torch.bfloat16
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=101 + sk)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale)
    o, lse = _run(gpu, q, k, v, scale)
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("sq", [1, 2, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_query_counts_and_dtypes(gpu, oracle_mod, sq, dtype):
    b, sk, h, d = 2, 200, 2, 32
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=211 + sq)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale)
    o, lse = _run(gpu, q, k, v, scale)
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("b,sq,h", [(48, 20, 4), (24, 1, 8), (48, 33, 4), (16, 64, 12), (48, 97, 4),
                                    (24, 150, 8), (48, 200, 4), (24, 256, 8), (32, 150, 6)])
@pytest.mark.parametrize("sk", [1, 37, 150, 256])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_grouped_heads(gpu, oracle_mod, b, sq, h, sk, dtype):
    """Head dim 16 with the heads in groups of four and more one-head tiles
    than SMs: items of one 32-row query block of four heads, the group's K
    and V loaded once for all of its blocks (one, two, several and ragged
    blocks per head, one key chunk to the most keys, several groups and
    batches); h = 6 takes the one-head-per-item path."""
    q, k, v = workloads.make_qkv(b, sq, sk, h, 16, dtype, seed=300 + sq + sk + h)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 0.25)
    o, lse = _run(gpu, q, k, v, 0.25)
    compare(o, lse, o_ref, lse_ref)


def test_grouped_heads_stay_apart(gpu, oracle_mod):
    """The four heads of a group share one 128-row tile but meet only their
    own keys and values: heads with scores and values of very different
    sizes side by side each match the oracle."""
    b, sq, sk, h, d = 48, 20, 90, 4, 16
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.float16, seed=77)
    k = k.float()
    v = v.float()
    k[:, :, 0] *= 8.0
    v[:, :, 1] *= 50.0
    k[:, :, 2] *= 0.05
    k, v = k.to(torch.float16), v.to(torch.float16)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 0.25)
    o, lse = _run(gpu, q, k, v, 0.25)
    # head 1's values are 50 times larger: its O tolerance scales with them
    compare(o[:, :, [0, 2, 3]], lse, o_ref[:, :, [0, 2, 3]], lse_ref)
    compare(o[:, :, 1:2] / 50.0, lse[:, 1:2], o_ref[:, :, 1:2] / 50.0, lse_ref[:, 1:2])


@pytest.mark.parametrize("scale", [0.0, -0.4, 1.3])
def test_scales(gpu, oracle_mod, scale):
    q, k, v = workloads.make_qkv(1, 140, 150, 4, 16, torch.float16, seed=5)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale)
    o, lse = _run(gpu, q, k, v, scale)
    compare(o, lse, o_ref, lse_ref)


def test_many_items_per_cta_both_kernels(gpu, oracle_mod):
    """b64 s150 h16 d16 fp16 (2048 tiles over the SMs): the short kernel and
    the general kernel both match the oracle on every row, and each other."""
    b, s, h, d = 64, 150, 16, 16
    q, k, v = workloads.make_qkv(b, s, s, h, d, torch.float16, seed=17)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale)
    o1, l1 = _run(gpu, q, k, v, scale)
    compare(o1, l1, o_ref, lse_ref)
    o2, l2 = _run(gpu, q, k, v, scale, general=True)
    compare(o2, l2, o_ref, lse_ref)
    assert (o1.float() - o2.float()).abs().max().item() <= 2e-2
    assert (l1 - l2).abs().max().item() <= 1e-3


def test_large_scores_stay_finite(gpu, oracle_mod):
    """Scores hundreds of units apart: the row max is taken before any
    exponential, so nothing overflows."""
    q, k, v = workloads.make_qkv(1, 130, 200, 2, 64, torch.bfloat16, seed=7)
    q = (q.float() * 6).to(torch.bfloat16)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 1.0)
    o, lse = _run(gpu, q, k, v, 1.0)
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("sk", [150, 256])
def test_increasing_scores_move_the_reference_max(gpu, oracle_mod, sk):
    """Keys whose scores grow by more than 8 (log2 units) from one pair of
    32-key chunks to the next: the reference max moves on every pair and the
    P already stored is rescaled each time."""
    b, sq, h, d = 1, 140, 2, 16
    q = torch.ones(b, sq, h, d).to(torch.float16)
    ramp = torch.linspace(0, 4, sk).view(1, sk, 1, 1)
    k = (ramp * torch.ones(b, sk, h, d)).to(torch.float16)
    _, _, v = workloads.make_qkv(b, sq, sk, h, d, torch.float16, seed=19)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 0.5)
    o, lse = _run(gpu, q, k, v, 0.5)
    compare(o, lse, o_ref, lse_ref)


def test_output_only_16_byte_aligned(gpu, oracle_mod):
    b, sq, sk, h, d = 1, 200, 100, 3, 16
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.float16, seed=43)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    n = q.numel()
    buf = torch.empty(n + 16, dtype=torch.float16, device="cuda")
    off = next(e for e in range(16) if (buf.data_ptr() + 2 * e) % 32 == 16)
    out = buf[off:off + n].view(q.shape)
    o, lse = gpu.attn_fwd(qd, kd, vd, out=out)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 1 / math.sqrt(d))
    compare(out, lse, o_ref, lse_ref)


@pytest.mark.parametrize("h", [2, 4])
def test_timeout_and_recovery(gpu, h):
    """ATTN_DEBUG_SKIP_LOADS: the producer issues nothing, the first wait on
    a full stage runs out after its bound, the kernel returns, the status
    reports it, and the next call works (h = 4: grouped items, whose copier
    warps wait on the same stages)."""
    b = 1 if h == 2 else 48  # h = 4, b = 48: 192 one-head tiles, so grouped items
    q, k, v = (t.cuda() for t in workloads.make_qkv(b, 64, 100, h, 16, torch.float16, seed=3))
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    gpu.attn_debug_set_flags(gpu.ATTN_DEBUG_SKIP_LOADS)
    try:
        gpu.attn_fwd(q, k, v)
    finally:
        gpu.attn_debug_set_flags(0)
    assert gpu.attn_get_device_status() == gpu.ATTN_ERR_DEVICE_TIMEOUT
    assert gpu.attn_last_timeout_site() >> 8 == 1
    o, lse = gpu.attn_fwd(q, k, v)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
