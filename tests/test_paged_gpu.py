"""Paged-KV decode parity: attn_decode_paged (through the C ABI) against the
fp64 oracle's paged reference.

A paged cache is only mentioned on the pages; the layout is the common one
(page pools [num_pages, page_size, h, d], an int32 block table per sequence,
int32 key counts on the device). Cases: shuffled pools, per-sequence lengths
that end mid-page and mid-block, one key, an empty sequence, a full table,
table entries past a sequence's end left as garbage (-1 and out-of-range
page numbers), pages whose stale rows hold NaN, explicit and heuristic
split counts, every head dim and both dtypes; page sizes from 16 keys up;
one new row per sequence (CUDA-core kernel) and several (tensor-core kernel,
with and without the causal mask aligned to each sequence's length).
"""
import math

import numpy as np
import pytest
import torch

import workloads
from parity import compare, to_np64

pytestmark = pytest.mark.gpu


def _make(b, h, d, page_size, max_pages, lens, dtype, seed, spare=3, sq=1):
    num_pages = b * max_pages + spare
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((b, sq, h, d), generator=g).to(dtype)
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


def _run(ea, oracle_mod, q, kp, vp, table, seqlens, splits, causal=False):
    d = q.shape[-1]
    o, lse = ea.attn_decode_paged(q.cuda(), kp.cuda(), vp.cuda(), table.cuda(), seqlens.cuda(),
                                  num_splits=splits, causal=causal)
    assert ea.attn_get_device_status() == ea.ATTN_OK
    # the oracle only reads used pages; give it a table with valid entries there
    o_ref, lse_ref = oracle_mod.paged_attention(q, kp, vp, table.numpy(), seqlens.numpy(),
                                                1 / math.sqrt(d), causal=causal)
    # rows that see no key (an empty sequence, or causal rows before its
    # first key) hold O = 0 and LSE = -inf exactly; the others are compared
    o64, l64 = to_np64(o), to_np64(lse)
    seen = np.isfinite(lse_ref)  # [b, h, sq]
    assert np.all(np.isneginf(l64[~seen]))
    assert np.all(o64.transpose(0, 2, 1, 3)[~seen] == 0.0)
    assert np.all(np.isfinite(l64[seen]))
    err_o = float(np.abs(o64 - o_ref).transpose(0, 2, 1, 3)[seen].max(initial=0.0))
    err_l = float(np.abs(l64[seen] - lse_ref[seen]).max(initial=0.0))
    assert err_o <= 2e-2, f"max |O - O_ref| = {err_o:.3e}"
    assert err_l <= 1e-3, f"max |LSE - LSE_ref| = {err_l:.3e}"


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


@pytest.mark.parametrize("page_size", [16, 48, 64, 128])
@pytest.mark.parametrize("d", [16, 128])
def test_paged_small_pages_one_row(gpu, oracle_mod, page_size, d):
    lens = [1, 15, 16, 17, 300, 64 * 17 + 5]
    max_pages = (max(lens) + page_size - 1) // page_size
    q, kp, vp, table, seqlens = _make(6, 3, d, page_size, max_pages, lens, torch.bfloat16,
                                      91 + page_size)
    for splits in (0, 1, 4):
        _run(gpu, oracle_mod, q, kp, vp, table, seqlens, splits)


@pytest.mark.parametrize("sq", [2, 10, 100, 300])
@pytest.mark.parametrize("page_size", [16, 64, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_paged_several_rows(gpu, oracle_mod, sq, page_size, causal):
    """Several new rows per sequence on the tensor-core kernel: 128-key tiles
    gathered from pages of 16, 64 or 256 keys; lengths that end mid-page
    (stale NaN rows in the last page must be zeroed before P V), below sq
    (causal rows that see nothing), and an empty sequence."""
    lens = [0, 5, 127, 128, 129, 1000, 2049]
    max_pages = (max(lens) + page_size - 1) // page_size
    q, kp, vp, table, seqlens = _make(7, 2, 128, page_size, max_pages, lens, torch.bfloat16,
                                      97 + sq, sq=sq)
    for splits in (0, 1, 3):
        _run(gpu, oracle_mod, q, kp, vp, table, seqlens, splits, causal=causal)


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_paged_several_rows_head_dims(gpu, oracle_mod, d, dtype):
    lens = [333, 64, 1]
    q, kp, vp, table, seqlens = _make(3, 3, d, 32, 12, lens, dtype, 103, sq=7)
    for causal in (False, True):
        _run(gpu, oracle_mod, q, kp, vp, table, seqlens, 2, causal=causal)


def test_paged_several_rows_match_contiguous_decode(gpu):
    """Identity table and full lengths: bit-identical to the contiguous
    several-row decode, with and without the causal mask."""
    b, sq, sk, h, d, ps = 2, 10, 4096, 8, 128, 64
    q, k, v = (t.cuda() for t in workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=107))
    kp = k.reshape(b * (sk // ps), ps, h, d)
    vp = v.reshape(b * (sk // ps), ps, h, d)
    table = torch.arange(b * (sk // ps), dtype=torch.int32, device="cuda").reshape(b, sk // ps)
    lens = torch.full((b,), sk, dtype=torch.int32, device="cuda")
    for causal in (False, True):
        for s in (1, 5):
            o1, l1 = gpu.attn_decode_splitkv(q, k, v, num_splits=s, causal=causal)
            o2, l2 = gpu.attn_decode_paged(q, kp, vp, table, lens, num_splits=s, causal=causal)
            assert gpu.attn_get_device_status() == gpu.ATTN_OK
            assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("causal", [False, True])
def test_paged_prefill_many_rows(gpu, oracle_mod, causal):
    """A chunk of many new rows per sequence from a paged cache (chunked
    prefill): 700 rows (three 256-row query blocks) over sequences of up to
    1500 keys in 64-key pages, through the same tensor-core path."""
    lens = [1500, 1111, 700]
    q, kp, vp, table, seqlens = _make(3, 4, 128, 64, 24, lens, torch.bfloat16, 109, sq=700)
    _run(gpu, oracle_mod, q, kp, vp, table, seqlens, 0, causal=causal)


def test_paged_rejects_unsupported_page_size(gpu):
    q = torch.zeros((1, 1, 1, 128), dtype=torch.bfloat16, device="cuda")
    kp = torch.zeros((2, 40, 1, 128), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    lens = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(gpu.AttnError):
        gpu.attn_decode_paged(q, kp, kp, table, lens)
