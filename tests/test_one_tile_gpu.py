"""Parity of the forward kernel compiled for at most 128 query rows (one live
query tile per unit, S double-buffered in TMEM so the next key tile's QK^T
runs while the softmax works on this one) against the fp64 oracle, through
the C ABI. It serves attn_fwd with sq <= 128 and more than 128 keys, and the
decode entry points with several new rows (key ranges and paged caches);
with at most 128 keys the two-tile kernel runs (the sk = 100 cases).

Cases: key-tile counts odd and even (1 to 6 tiles, ragged last tiles), one to
128 rows, every head dim and both dtypes, key ranges (explicit and heuristic
splits), the causal mask, paged caches, many units per CTA, and keys whose
scores grow tile after tile so the reference max moves on every tile and the
O rescale (which waits for the previous tile's P V) runs each time.
Tolerance as everywhere: max |O - O_ref| <= 2e-2, max |LSE - LSE_ref| <= 1e-3.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from parity import compare, compare_masked, to_np64

pytestmark = pytest.mark.gpu


def _fwd(ea, q, k, v, scale, causal=False):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = ea.attn_fwd(qd, kd, vd, scale=scale, causal=causal)
    assert ea.attn_get_device_status() == ea.ATTN_OK
    return o, lse


def _decode(ea, q, k, v, scale, splits, causal=False):
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = ea.attn_decode_splitkv(qd, kd, vd, scale=scale, num_splits=splits, causal=causal)
    assert ea.attn_get_device_status() == ea.ATTN_OK
    return o, lse


def _ramp_keys(b, sq, sk, h, d, dtype, seed):
    """Q all ones, K rows growing with their index: each key tile's scores
    exceed the last one's, by more than the lazy threshold at scale 0.5."""
    q = torch.ones(b, sq, h, d).to(dtype)
    ramp = torch.linspace(0, 4, sk).view(1, sk, 1, 1)
    k = (ramp * torch.ones(b, sk, h, d)).to(dtype)
    _, _, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=seed)
    return q, k, v


@pytest.mark.parametrize("sq", [1, 10, 77, 128])
@pytest.mark.parametrize("sk", [100, 129, 256, 300, 640, 700])
def test_key_tile_counts(gpu, oracle_mod, sq, sk):
    b, h, d = 2, 3, 128
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=301 + sq + sk)
    scale = 1 / math.sqrt(d)
    o, lse = _fwd(gpu, q, k, v, scale)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale)
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_head_dims_and_dtypes(gpu, oracle_mod, d, dtype):
    b, sq, sk, h = 1, 100, 700, 3
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=311 + d)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale)
    o, lse = _fwd(gpu, q, k, v, scale)
    compare(o, lse, o_ref, lse_ref)
    for splits in (0, 3):
        o, lse = _decode(gpu, q, k, v, scale, splits)
        compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("sq", [10, 128])
def test_rescale_every_tile_plain_and_key_ranges(gpu, oracle_mod, sq):
    b, sk, h, d = 1, 1024, 2, 64
    q, k, v = _ramp_keys(b, sq, sk, h, d, torch.bfloat16, seed=321)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 0.5)
    o, lse = _fwd(gpu, q, k, v, 0.5)
    compare(o, lse, o_ref, lse_ref)
    for splits in (0, 2, 3):
        o, lse = _decode(gpu, q, k, v, 0.5, splits)
        compare(o, lse, o_ref, lse_ref)


def test_rescale_every_tile_causal(gpu, oracle_mod):
    b, sq, sk, h, d = 1, 100, 900, 2, 128
    q, k, v = _ramp_keys(b, sq, sk, h, d, torch.bfloat16, seed=331)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, 0.5, causal=True)
    o, lse = _fwd(gpu, q, k, v, 0.5, causal=True)
    compare_masked(o, lse, o_ref, lse_ref)
    o, lse = _decode(gpu, q, k, v, 0.5, 3, causal=True)
    compare_masked(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_rescale_every_tile_paged(gpu, oracle_mod, causal):
    """The ramp cache cut into shuffled 64-key pages behind a block table,
    sequences of different lengths, ten new rows each."""
    b, sq, h, d, ps = 2, 10, 2, 128, 64
    lens = [1000, 613]
    max_pages = 16
    q, k, v = _ramp_keys(b, sq, ps * max_pages, h, d, torch.bfloat16, seed=341)
    num_pages = b * max_pages
    perm = torch.randperm(num_pages, generator=torch.Generator().manual_seed(7))
    kp = torch.empty((num_pages, ps, h, d), dtype=k.dtype)
    vp = torch.empty_like(kp)
    kp[perm] = k.reshape(num_pages, ps, h, d)
    vp[perm] = v.reshape(num_pages, ps, h, d)
    table = perm.to(torch.int32).reshape(b, max_pages).contiguous()
    seqlens = torch.tensor(lens, dtype=torch.int32)
    o, lse = gpu.attn_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), seqlens.cuda(),
                                   scale=0.5, causal=causal)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    o_ref, lse_ref = oracle_mod.paged_attention(q, kp, vp, table.numpy(), seqlens.numpy(), 0.5,
                                                causal=causal)
    o64, l64 = to_np64(o), to_np64(lse)
    assert np.abs(o64 - o_ref).max() <= 2e-2
    assert np.abs(l64 - lse_ref).max() <= 1e-3


@pytest.mark.parametrize("splits", [1, 4])
def test_many_units_per_cta(gpu, oracle_mod, splits):
    """b16 h32 with 16 new rows: 512 units (2048 with four key ranges) over
    the SMs, so every CTA runs several units back to back through both S
    buffers and the O accumulator; every row is compared."""
    b, sq, sk, h, d = 16, 16, 700, 32, 128
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=351)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale)
    o, lse = _decode(gpu, q, k, v, scale, splits)
    compare(o, lse, o_ref, lse_ref)


def test_one_and_two_tile_kernels_agree(gpu):
    """The same 128 query rows through the one-tile kernel (sq = 128) and as
    the first rows of a 129-row call (the two-tile kernel): identical keys,
    so identical arithmetic row by row."""
    b, sk, h, d = 2, 900, 4, 128
    q, k, v = workloads.make_qkv(b, 129, sk, h, d, torch.bfloat16, seed=361)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o2, l2 = gpu.attn_fwd(qd, kd, vd)
    o1, l1 = gpu.attn_fwd(qd[:, :128].contiguous(), kd, vd)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    assert torch.equal(o1, o2[:, :128])
    assert torch.equal(l1, l2[:, :, :128])
