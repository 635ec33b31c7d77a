"""Paged-KV decode parity: attn_decode_paged (through the C ABI) against the
fp64 oracle's paged reference.

A paged cache is only mentioned on the pages; the layout is the common one
(page pools [num_pages, page_size, h, d], an int32 block table per sequence,
int32 key counts on the device). Cases: shuffled pools, per-sequence lengths
that end mid-page and mid-block, one key, an empty sequence, a full table,
table entries past a sequence's end left as garbage (-1 and out-of-range
page numbers), pages whose stale rows hold NaN, explicit and heuristic
split counts, every head dim and both dtypes.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from parity import compare, to_np64

pytestmark = pytest.mark.gpu


def _make(b, h, d, page_size, max_pages, lens, dtype, seed, spare=3):
    num_pages = b * max_pages + spare
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((b, 1, h, d), generator=g).to(dtype)
    kp = torch.randn((num_pages, page_size, h, d), generator=g).to(dtype)
    vp = torch.randn((num_pages, page_size, h, d), generator=g).to(dtype)
    perm = torch.randperm(num_pages, generator=g)[: b * max_pages].reshape(b, max_pages)
    table = perm.to(torch.int32).clone()
    for i, n in enumerate(lens):  # entries past the sequence's last page are never read
        used = (n + page_size - 1) // page_size
        if used < max_pages:
            table[i, used:] = torch.tensor([-1, 10 ** 6, num_pages][: max_pages - used] +
                                           [-1] * max(0, max_pages - used - 3), dtype=torch.int32)
    # stale rows past each sequence's end in its last page: NaN must not reach O
    for i, n in enumerate(lens):
        if n % page_size and n > 0:
            pg = int(table[i, n // page_size])
            vp[pg, n % page_size:] = float("nan")
            kp[pg, n % page_size:] = float("nan")
    seqlens = torch.tensor(lens, dtype=torch.int32)
    return q, kp, vp, table, seqlens


def _run(ea, oracle_mod, q, kp, vp, table, seqlens, splits):
    d = q.shape[-1]
    o, lse = ea.attn_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), seqlens.cuda(),
                                  num_splits=splits)
    assert ea.attn_get_device_status() == ea.ATTN_OK
    # the oracle only reads used pages; give it a table with valid entries there
    o_ref, lse_ref = oracle_mod.paged_attention(q, kp, vp, table.numpy(), seqlens.numpy(),
                                                1 / math.sqrt(d))
    lens = seqlens.numpy()
    nz = [i for i in range(len(lens)) if lens[i] > 0]
    if len(nz) < len(lens):
        z = [i for i in range(len(lens)) if lens[i] == 0]
        assert np.all(to_np64(o)[z] == 0.0) and np.all(np.isneginf(to_np64(lse)[z]))
    compare(o[nz], lse[nz], o_ref[nz], lse_ref[nz])


@pytest.mark.parametrize("splits", [0, 1, 3, 17])
def test_paged_lengths_and_splits(gpu, oracle_mod, splits):
    lens = [1, 256, 300, 1000, 4096, 2049]
    q, kp, vp, table, seqlens = _make(6, 4, 128, 256, 16, lens, torch.bfloat16, 81)
    _run(gpu, oracle_mod, q, kp, vp, table, seqlens, splits)


def test_paged_empty_and_full_sequences(gpu, oracle_mod):
    lens = [0, 8 * 512, 513]
    q, kp, vp, table, seqlens = _make(3, 2, 128, 512, 8, lens, torch.bfloat16, 83)
    for splits in (0, 1, 5):
        _run(gpu, oracle_mod, q, kp, vp, table, seqlens, splits)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_paged_head_dims_and_dtypes(gpu, oracle_mod, d, dtype):
    lens = [700, 1, 3 * 256]
    q, kp, vp, table, seqlens = _make(3, 3, d, 256, 5, lens, dtype, 87)
    for splits in (0, 2):
        _run(gpu, oracle_mod, q, kp, vp, table, seqlens, splits)


def test_paged_matches_contiguous_decode(gpu):
    """Identity table and full lengths: the same result as the contiguous
    split decode on the same cache."""
    b, sk, h, d, ps = 2, 4096, 8, 128, 256
    q, k, v = (t.cuda() for t in workloads.make_qkv(b, 1, sk, h, d, torch.bfloat16, seed=89))
    kp = k.reshape(b * (sk // ps), ps, h, d)
    vp = v.reshape(b * (sk // ps), ps, h, d)
    table = torch.arange(b * (sk // ps), dtype=torch.int32, device="cuda").reshape(b, sk // ps)
    lens = torch.full((b,), sk, dtype=torch.int32, device="cuda")
    for s in (1, 4):
        o1, l1 = gpu.attn_decode_splitkv(q, k, v, num_splits=s)
        o2, l2 = gpu.attn_decode_paged(q, kp, vp, table, lens, num_splits=s)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_paged_rejects_unsupported_page_size(gpu):
    q = torch.zeros((1, 1, 1, 128), dtype=torch.bfloat16, device="cuda")
    kp = torch.zeros((2, 128, 1, 128), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(gpu.AttnError):
        gpu.attn_decode_paged(q, kp, kp, table, lens)
