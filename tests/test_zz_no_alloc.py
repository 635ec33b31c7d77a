"""The decode entry point that allocates nothing.

attn_decode_splitkv_noalloc serves callers that cannot allocate device memory
once they run (memory owned by their own allocator or pool, a fixed memory
budget, real-time code that forbids allocation after start-up): its per-split
partials live in a fixed array inside the library instead of the device's
memory pool. It must give what the allocating entry point
(attn_decode_splitkv_ex) gives, and what the fp64 oracle gives, within the
tolerances of the other parity tests, on consecutive calls that share the
array; it must refuse, before launching anything, a request whose partials do
not fit; and a bounded wait that runs out in its kernels must reach the
caller through its own status reader, which allocates nothing either.

This file is named so that pytest collects it last.
"""
import ctypes
import math
import time

import pytest
import torch

import workloads
from parity import LSE_TOL, O_TOL, compare

pytestmark = pytest.mark.gpu


def _raw_noalloc(lib, q, k, v, o, lse, scale, splits, dtype_code):
    fn = lib.attn_decode_splitkv_noalloc
    fn.restype = ctypes.c_int
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32, i32, vp]
    b, sq, h, d = q.shape
    sk = k.shape[1]
    return fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), b, sq, sk, h,
              d, scale, splits, dtype_code, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _raw_status(lib):
    fn = lib.attn_get_noalloc_status
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p]
    return fn(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("b,sq,sk,h,d,dtype,splits", [
    (1, 1, 32768, 16, 128, torch.bfloat16, 0),   # the b1 h16 sk32768 decode, heuristic splits
    (2, 3, 3000, 4, 64, torch.float16, 5),       # several query rows, fp16, explicit splits
    (1, 1, 310, 2, 128, torch.bfloat16, 4),      # an empty split
    (8, 1, 8192, 48, 128, torch.bfloat16, 0),    # the heuristic picks one split: no scratch
    (1, 2, 5000, 3, 16, torch.float16, 0),       # several rows on the tensor-core kernel ...
    (1, 5, 5000, 3, 16, torch.bfloat16, 3),
    (2, 10, 4000, 2, 128, torch.bfloat16, 0),
    (1, 10, 4000, 5, 128, torch.float16, 3),
    (1, 5, 300, 2, 128, torch.bfloat16, 40),     # ... a count lowered to the 3 key tiles
])
def test_matches_allocating_entry_point_and_oracle_on_two_calls(gpu, oracle_mod, b, sq, sk, h, d,
                                                                dtype, splits):
    lib = gpu.load_library()
    hq, hk, hv = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=41)
    q, k, v = (t.cuda() for t in (hq, hk, hv))
    scale = 1.0 / math.sqrt(d)
    ref_o, ref_lse = gpu.attn_decode_splitkv(q, k, v, scale=scale, num_splits=splits)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    o_ref, lse_ref = oracle_mod.attention(hq, hk, hv, scale)
    code = gpu.ATTN_BF16 if dtype == torch.bfloat16 else gpu.ATTN_FP16
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((b, h, sq), float("nan"), dtype=torch.float32, device="cuda")
        assert _raw_noalloc(lib, q, k, v, o, lse, scale, splits, code) == gpu.ATTN_OK
        assert _raw_status(lib) == gpu.ATTN_OK
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert (o.float() - ref_o.float()).abs().max().item() <= O_TOL
        assert (lse - ref_lse).abs().max().item() <= LSE_TOL
        compare(o, lse, o_ref, lse_ref)


def test_rejects_requests_larger_than_the_array(gpu):
    lib = gpu.load_library()
    b, sq, sk, h, d = 8, 1, 8192, 48, 128
    # 64 splits of 384 rows need 64 * 384 * 129 * 4 bytes, more than the array holds
    assert 64 * b * sq * h * (d + 1) * 4 > (8 << 20)
    q = torch.zeros(b, sq, h, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(b, sk, h, d, dtype=torch.bfloat16, device="cuda")
    o = torch.full_like(q, 7.0)
    lse = torch.full((b, h, sq), 7.0, dtype=torch.float32, device="cuda")
    rc = _raw_noalloc(lib, q, k, k, o, lse, 0.1, 64, gpu.ATTN_BF16)
    assert rc == gpu.ATTN_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())  # nothing was launched


@pytest.mark.parametrize("sq,kernel", [(1, 2), (5, 1)])
def test_timeout_reaches_its_status_reader_and_the_context_recovers(gpu, sq, kernel):
    """The failure is made on the host: ATTN_DEBUG_SKIP_LOADS makes the
    producers issue no copy, so the first wait on a "full" barrier runs out
    after its bound (about two seconds) and the kernel returns. sq = 1 runs
    the CUDA-core split kernel (kernel code 2), sq = 5 the tensor-core
    forward kernel (kernel code 1)."""
    lib = gpu.load_library()
    b, sk, h, d = 1, 4096, 2, 128
    q, k, v = (t.cuda() for t in workloads.make_qkv(b, sq, sk, h, d, torch.bfloat16, seed=43))
    o = torch.empty_like(q)
    lse = torch.empty((b, h, sq), dtype=torch.float32, device="cuda")
    assert _raw_status(lib) == gpu.ATTN_OK
    gpu.attn_debug_set_flags(gpu.ATTN_DEBUG_SKIP_LOADS)
    try:
        rc = _raw_noalloc(lib, q, k, v, o, lse, 1 / math.sqrt(d), 2, gpu.ATTN_BF16)
    finally:
        gpu.attn_debug_set_flags(0)
    assert rc == gpu.ATTN_OK
    t0 = time.time()
    assert _raw_status(lib) == gpu.ATTN_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 60
    assert gpu.attn_last_timeout_site() >> 8 == kernel
    # cleared, and the main status word was not touched
    assert _raw_status(lib) == gpu.ATTN_OK
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    ref_o, ref_lse = gpu.attn_decode_splitkv(q, k, v, num_splits=2)
    assert _raw_noalloc(lib, q, k, v, o, lse, 1 / math.sqrt(d), 2, gpu.ATTN_BF16) == gpu.ATTN_OK
    assert _raw_status(lib) == gpu.ATTN_OK
    assert (o.float() - ref_o.float()).abs().max().item() <= O_TOL
    assert (lse - ref_lse).abs().max().item() <= LSE_TOL
