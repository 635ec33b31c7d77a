"""The decode entry point that allocates nothing.

attn_decode_splitkv_noalloc serves callers that cannot allocate device memory
once they run (memory owned by their own allocator or pool, a fixed memory
budget, real-time code that forbids allocation after start-up): its per-split
partials live in a fixed array inside the library instead of the device's
memory pool. It must give what the allocating entry point
(attn_decode_splitkv_ex) gives, within the tolerances of the other parity
tests, on consecutive calls that share the array; and it must refuse, before
launching anything, a request whose partials do not fit.

This file is named so that pytest collects it last.
"""
import ctypes
import math

import pytest
import torch

import workloads
from parity import LSE_TOL, O_TOL

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


@pytest.mark.parametrize("b,sq,sk,h,d,dtype,splits", [
    (1, 1, 32768, 16, 128, torch.bfloat16, 0),   # the b1 h16 sk32768 decode, heuristic splits
    (2, 3, 3000, 4, 64, torch.float16, 5),       # several query rows, fp16, explicit splits
    (1, 1, 310, 2, 128, torch.bfloat16, 4),      # an empty split
    (8, 1, 8192, 48, 128, torch.bfloat16, 0),    # the heuristic picks one split: no scratch
])
def test_matches_allocating_entry_point_on_two_calls(gpu, b, sq, sk, h, d, dtype, splits):
    lib = gpu.load_library()
    q, k, v = (t.cuda() for t in workloads.make_qkv(b, sq, sk, h, d, dtype, seed=41))
    scale = 1.0 / math.sqrt(d)
    ref_o, ref_lse = gpu.attn_decode_splitkv(q, k, v, scale=scale, num_splits=splits)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    code = gpu.ATTN_BF16 if dtype == torch.bfloat16 else gpu.ATTN_FP16
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((b, h, sq), float("nan"), dtype=torch.float32, device="cuda")
        assert _raw_noalloc(lib, q, k, v, o, lse, scale, splits, code) == gpu.ATTN_OK
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        assert (o.float() - ref_o.float()).abs().max().item() <= O_TOL
        assert (lse - ref_lse).abs().max().item() <= LSE_TOL


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
