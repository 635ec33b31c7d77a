"""Maximum sizes: K and V with 2^31 elements each (b1, 2^20 keys, h16, d128:
4 GiB apiece in bf16), so every element offset into them, and into dK and
dV, passes 2^31 - 1, through the forward kernels (one and two query tiles),
the one-row and several-row decode and the backward tile kernels.

The oracle cannot hold those tensors in fp64, so the keys repeat a pattern:
K and V are a 256-key block repeated m = 4096 times. Attention over keys that
each appear m times is attention over one block with every weight taken m
times, which the normalisation cancels (a closed form of the definition, for
any m):
    O = O_block,   LSE = LSE_block + ln m,
    dQ = dQ_block, dK_j = dK_block(j mod 256) / m, dV_j = dV_block(j mod 256) / m,
where *_block is the oracle on the one 256-key block. dK and dV are compared
after multiplying by m (their 16-bit values keep their relative precision).
Tolerances as everywhere: 2e-2 on O, 1e-3 on LSE, 2e-2 (1 + max |ref|) on
gradients.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from parity import compare, to_np64

pytestmark = pytest.mark.gpu

BLOCK, REPS, H, D = 256, 4096, 16, 128
SK = BLOCK * REPS  # 2^20 keys: 2^31 elements per K / V


@pytest.fixture(scope="module")
def big(gpu):
    torch.cuda.empty_cache()
    _, kb, vb = workloads.make_qkv(1, 1, BLOCK, H, D, torch.bfloat16, seed=501)
    k = kb.cuda().repeat(1, REPS, 1, 1)
    v = vb.cuda().repeat(1, REPS, 1, 1)
    assert k.numel() == 2 ** 31 and k.is_contiguous()
    yield kb, vb, k, v
    del k, v
    torch.cuda.empty_cache()


def _block_ref(oracle_mod, q, kb, vb, scale):
    o_ref, lse_ref = oracle_mod.attention(q, kb, vb, scale)
    return o_ref, lse_ref + math.log(REPS)


@pytest.mark.parametrize("sq", [1, 100, 300])
def test_forward(gpu, oracle_mod, big, sq):
    """sq = 1 and 100: the one-tile forward kernel; 300: two query tiles per
    unit and a ragged one."""
    kb, vb, k, v = big
    q, _, _ = workloads.make_qkv(1, sq, 1, H, D, torch.bfloat16, seed=502 + sq)
    scale = 1 / math.sqrt(D)
    o, lse = gpu.attn_fwd(q.cuda(), k, v, scale=scale)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    o_ref, lse_ref = _block_ref(oracle_mod, q, kb, vb, scale)
    compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("sq,splits", [(1, 0), (1, 16), (4, 0), (10, 7)])
def test_decode(gpu, oracle_mod, big, sq, splits):
    """One new row (the CUDA-core split kernel) and several (the one-tile
    forward kernel over key ranges), heuristic and explicit split counts."""
    kb, vb, k, v = big
    q, _, _ = workloads.make_qkv(1, sq, 1, H, D, torch.bfloat16, seed=512 + sq)
    scale = 1 / math.sqrt(D)
    o, lse = gpu.attn_decode_splitkv(q.cuda(), k, v, scale=scale, num_splits=splits)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    o_ref, lse_ref = _block_ref(oracle_mod, q, kb, vb, scale)
    compare(o, lse, o_ref, lse_ref)


def test_backward(gpu, oracle_mod, big):
    """The key-tile and query-tile kernels over 8192 key tiles per head;
    dK and dV hold 2^31 elements each."""
    kb, vb, k, v = big
    sq = 200
    q, _, _ = workloads.make_qkv(1, sq, 1, H, D, torch.bfloat16, seed=521)
    do = torch.randn((1, sq, H, D), generator=torch.Generator().manual_seed(522)).to(
        torch.bfloat16)
    scale = 1 / math.sqrt(D)
    qd, dod = q.cuda(), do.cuda()
    o, lse = gpu.attn_fwd(qd, k, v, scale=scale)
    dq, dk, dv = gpu.attn_bwd(qd, k, v, o, lse, dod, scale=scale)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    rq, rk, rv = oracle_mod.attention_backward(q, kb, vb, do, scale)
    got_q = to_np64(dq)
    assert np.abs(got_q - rq).max() <= 2e-2 * (1.0 + np.abs(rq).max())
    # every key row equals its block row / m: check the first and last blocks
    # whole, and every block's row 0 and row 255 (as m times the value)
    for name, g, r in (("dk", dk, rk), ("dv", dv, rv)):
        g = g.view(1, REPS, BLOCK, H, D)
        bound = 2e-2 * (1.0 + float(np.abs(r).max()))
        for blk in (0, REPS - 1):
            err = float(np.abs(to_np64(g[:, blk]) * REPS - r).max())
            assert err <= bound, f"{name} block {blk}: {err:.3e} > {bound:.3e}"
        for row in (0, BLOCK - 1):
            got = to_np64(g[0, :, row]) * REPS  # [REPS, H, D]
            err = float(np.abs(got - r[0, row][None]).max())
            assert err <= bound, f"{name} row {row} of every block: {err:.3e} > {bound:.3e}"
