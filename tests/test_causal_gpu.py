"""Causal forward and decode parity: the CUDA path (through the C ABI)
against the fp64 oracle's causal reading.

Causal masking is not on the pages; the reading (oracle and kernels alike)
is the bottom-right-aligned mask: query row i of sq sees key j of sk only if
j <= i + sk - sq. Rows that see no key (sq > sk) give O = 0 and
LSE = -inf. Shapes cover sq == sk (tile edges and ragged tails), sq < sk
(new rows appended to a cache, through the forward and the split decode),
sq > sk, every head dim and both dtypes. Tolerance as everywhere: max |O -
O_ref| <= 2e-2, max |LSE - LSE_ref| <= 1e-3 on rows that see a key.
"""
import math

import pytest
import torch

import workloads
from parity import compare_masked

pytestmark = pytest.mark.gpu


def _inputs(b, sq, sk, h, d, dtype, seed):
    return workloads.make_qkv(b, sq, sk, h, d, dtype, seed=seed)


def _check(ea, oracle_mod, q, k, v, scale, o, lse, rows=None):
    assert ea.attn_get_device_status() == ea.ATTN_OK
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale, rows=rows, causal=True)
    compare_masked(o, lse, o_ref, lse_ref, rows=rows)


@pytest.mark.parametrize("b,s,h,d", [(2, 300, 3, 128), (1, 64, 2, 16), (1, 1000, 2, 64),
                                     (2, 129, 2, 32), (1, 256, 4, 128), (1, 257, 1, 128)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_causal_square(gpu, oracle_mod, b, s, h, d, dtype):
    q, k, v = _inputs(b, s, s, h, d, dtype, 61)
    scale = 1 / math.sqrt(d)
    o, lse = gpu.attn_fwd(*(t.cuda() for t in (q, k, v)), causal=True)
    _check(gpu, oracle_mod, q, k, v, scale, o, lse)


@pytest.mark.parametrize("sq,sk", [(200, 700), (10, 3000), (1, 500), (127, 128), (300, 100),
                                   (5, 1)])
def test_causal_rectangular_forward(gpu, oracle_mod, sq, sk):
    b, h, d = 2, 2, 128
    q, k, v = _inputs(b, sq, sk, h, d, torch.bfloat16, 67)
    o, lse = gpu.attn_fwd(*(t.cuda() for t in (q, k, v)), causal=True)
    _check(gpu, oracle_mod, q, k, v, 1 / math.sqrt(d), o, lse)


@pytest.mark.parametrize("sq,sk", [(10, 3000), (2, 20000), (300, 5000), (16, 129)])
@pytest.mark.parametrize("splits", [0, 1, 4, 40])
def test_causal_split_decode(gpu, oracle_mod, sq, sk, splits):
    """New rows appended to a cache: later splits cover keys that some of
    the new rows may not see yet."""
    b, h, d = 1, 3, 128
    q, k, v = _inputs(b, sq, sk, h, d, torch.bfloat16, 71)
    o, lse = gpu.attn_decode_splitkv(*(t.cuda() for t in (q, k, v)), num_splits=splits,
                                     causal=True)
    _check(gpu, oracle_mod, q, k, v, 1 / math.sqrt(d), o, lse)


def test_causal_decode_one_row_is_unmasked(gpu):
    b, sk, h, d = 2, 5000, 4, 128
    q, k, v = (t.cuda() for t in _inputs(b, 1, sk, h, d, torch.bfloat16, 73))
    o0, l0 = gpu.attn_decode_splitkv(q, k, v)
    o1, l1 = gpu.attn_decode_splitkv(q, k, v, causal=True)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_causal_mid_shape_all_rows(gpu, oracle_mod):
    w = workloads.WORKLOADS["mid_fwd"]
    q, k, v = workloads.make_workload(w)
    o, lse = gpu.attn_fwd(*(t.cuda() for t in (q, k, v)), causal=True)
    _check(gpu, oracle_mod, q, k, v, w.scale, o, lse)


def test_causal_several_units_per_cta_all_rows(gpu, oracle_mod):
    """More causal units than SMs (b2 s1024 h48: 384 units dealt longest
    first over 152 CTAs); every row is compared."""
    b, s, h, d = 2, 1024, 48, 128
    q, k, v = _inputs(b, s, s, h, d, torch.bfloat16, 79)
    o, lse = gpu.attn_fwd(*(t.cuda() for t in (q, k, v)), causal=True)
    _check(gpu, oracle_mod, q, k, v, 1 / math.sqrt(d), o, lse)
