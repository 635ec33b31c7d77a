"""exact_attention_65_gb300: exact attention on one GB300 through the exattn C ABI.

A thin ctypes binding over ``libexattn.so`` (built by
``exact_attention_65_gb300.build``). It only checks and marshals arguments:
every step of the computation runs in the library's CUDA kernels, and there
is no CPU or framework fallback. PyTorch supplies device memory and the
current CUDA stream.

    o, lse = attn_fwd(q, k, v)                  # q, k, v: [b, s, h, d] fp16/bf16 CUDA tensors
    o, lse = attn_decode_splitkv(q, k, v)       # split-KV decode, num_splits=0: heuristic
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libexattn.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "exattn.h")

ATTN_FP16, ATTN_BF16 = 0, 1
ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_NO_MEMORY = 4
ATTN_ERR_DEVICE_TIMEOUT = 5
ATTN_DEBUG_SKIP_LOADS = 1
ATTN_DEBUG_GENERAL_FWD = 2
ATTN_DEBUG_GENERAL_BWD = 4

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    """A non-OK status returned by the C ABI."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} (status {status})")


def load_library() -> ctypes.CDLL:
    """Load libexattn.so; raise if it has not been built (there is no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m exact_attention_65_gb300.build` (there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, f32, u32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint
        lib.attn_fwd.restype = i32
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp]
        lib.attn_decode_splitkv.restype = i32
        lib.attn_decode_splitkv.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp]
        lib.attn_decode_splitkv_ex.restype = i32
        lib.attn_decode_splitkv_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32,
                                               i32, i32, vp]
        lib.attn_fwd_host.restype = i32
        lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, i32, vp]
        lib.attn_fwd_causal.restype = i32
        lib.attn_fwd_causal.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp]
        lib.attn_decode_splitkv_causal.restype = i32
        lib.attn_decode_splitkv_causal.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                   f32, i32, i32, vp]
        lib.attn_decode_paged.restype = i32
        lib.attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                          i32, f32, i32, i32, vp]
        lib.attn_decode_paged_ex.restype = i32
        lib.attn_decode_paged_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                             i32, i32, f32, i32, i32, i32, vp]
        for fn in (lib.attn_bwd, lib.attn_bwd_causal):
            fn.restype = i32
            fn.argtypes = [vp] * 9 + [i32, i32, i32, i32, i32, f32, i32, vp]
        lib.attn_decode_splitkv_noalloc.restype = i32
        lib.attn_decode_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32,
                                                    f32, i32, i32, vp]
        lib.attn_get_noalloc_status.restype = i32
        lib.attn_get_noalloc_status.argtypes = [vp]
        lib.attn_decode_num_splits.restype = i32
        lib.attn_decode_num_splits.argtypes = [i32] * 5
        lib.attn_decode_num_splits_for_sms.restype = i32
        lib.attn_decode_num_splits_for_sms.argtypes = [i32] * 6
        lib.attn_get_device_status.restype = i32
        lib.attn_get_device_status.argtypes = [vp]
        lib.attn_last_timeout_site.restype = u32
        lib.attn_last_timeout_site.argtypes = []
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_status_string.argtypes = [i32]
        lib.attn_release_workspace.restype = None
        lib.attn_release_workspace.argtypes = []
        lib.attn_debug_set_flags.restype = None
        lib.attn_debug_set_flags.argtypes = [u32]
        lib.attn_version.restype = i32
        lib.attn_version.argtypes = []
        _lib = lib
        return lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


_DTYPE_CODE = {torch.float16: ATTN_FP16, torch.bfloat16: ATTN_BF16}
_current_raw_stream = torch._C._cuda_getCurrentRawStream
_current_device = torch._C._cuda_getDevice


def _dtype_code(t: torch.Tensor) -> int:
    code = _DTYPE_CODE.get(t.dtype)
    if code is None:
        raise TypeError(f"exattn takes float16 or bfloat16 tensors, got {t.dtype}")
    return code


def _check_slow(q, k, v):
    """Raises the specific error for a q, k, v triple _check refused."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [b, s, h, d], got shape {tuple(t.shape)}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous in (b, s, h, d) order")
    raise ValueError("invalid q, k, v")


def _check(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    """Sizes (b, sq, sk, h, d), dtype code and device index of a q, k, v
    triple; raises on anything the C ABI would not take. Kept lean: small
    problems issue in a few microseconds, and this runs on every call."""
    try:
        ok = (q.is_cuda and k.is_cuda and v.is_cuda and q.dim() == 4 and k.dim() == 4
              and v.dim() == 4 and q.is_contiguous() and k.is_contiguous() and v.is_contiguous())
    except AttributeError:
        ok = False
    if not ok:
        _check_slow(q, k, v)
    dt = q.dtype
    if k.dtype is not dt or v.dtype is not dt:
        raise TypeError("q, k, v must share one dtype")
    idx = q.get_device()
    if k.get_device() != idx or v.get_device() != idx:
        raise ValueError("q, k, v must be on the same device")
    b, sq, h, d = q.shape
    kb, sk, kh, kd = k.shape
    if kb != b or kh != h or kd != d or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    code = _DTYPE_CODE.get(dt)
    if code is None:
        raise TypeError(f"exattn takes float16 or bfloat16 tensors, got {dt}")
    return b, sq, sk, h, d, code, idx


def _outputs(q, out, lse, b, h, sq, idx):
    if out is None:
        out = torch.empty_like(q)
    elif (out.shape != q.shape or out.dtype is not q.dtype or not out.is_contiguous()
          or out.get_device() != idx):
        raise ValueError("out must be a contiguous tensor like q")
    if lse is None:
        lse = torch.empty((b, h, sq), dtype=torch.float32, device=q.device)
    elif (lse.shape != (b, h, sq) or lse.dtype is not torch.float32 or not lse.is_contiguous()
          or lse.get_device() != idx):
        raise ValueError("lse must be a contiguous float32 tensor [b, h, sq]")
    return out, lse


def _stream(device, stream):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _call(fn, idx, stream, *args):
    """Call C-ABI function ``fn`` with ``args`` plus the stream, with device
    ``idx`` current. The common case (device already current, its current
    stream) skips the device context manager and the Stream object."""
    if idx == _current_device():
        raw = _current_raw_stream(idx) if stream is None else stream.cuda_stream
        return fn(*args, raw)
    device = torch.device("cuda", idx)
    with torch.cuda.device(device):
        return fn(*args, _stream(device, stream))


def attn_fwd(q, k, v, scale: float | None = None, out=None, lse=None, stream=None,
             causal: bool = False):
    """Exact attention O = softmax(scale * Q K^T) V and LSE [b, h, sq] (fp32).

    q: [b, sq, h, d], k/v: [b, sk, h, d], fp16 or bf16, contiguous CUDA
    tensors; default scale 1/sqrt(d). Runs on ``stream`` (default: the
    current stream of q's device). ``causal``: bottom-right-aligned mask
    (query row i sees key j only if j <= i + sk - sq)."""
    b, sq, sk, h, d, dt, idx = _check(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out, lse = _outputs(q, out, lse, b, h, sq, idx)
    lib = _lib or load_library()
    fn = lib.attn_fwd_causal if causal else lib.attn_fwd
    rc = _call(fn, idx, stream, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
               lse.data_ptr(), b, sq, sk, h, d, scale, dt)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_fwd_causal" if causal else "attn_fwd")
    return out, lse


def attn_fwd_host(q, k, v, scale: float | None = None, out=None, lse=None, causal: bool = False,
                  device=None, stream=None, sync: bool = True):
    """attn_fwd on host (CPU) tensors through the library's copy / compute /
    copy-back pipeline (attn_fwd_host in the C ABI).

    q: [b, sq, h, d], k/v: [b, sk, h, d], fp16 or bf16, contiguous CPU
    tensors, best in pinned memory (pageable ones work, without overlap).
    out and lse (CPU) are allocated pinned when not given. Runs on
    ``device`` (default: the current CUDA device) and ``stream`` (its
    current stream). With ``sync`` False the call returns once the work is
    queued: out and lse are valid, and the inputs may be reused, only after
    the stream is synchronised."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
            raise ValueError(f"{name} must be a CPU tensor (attn_fwd takes CUDA tensors)")
        if t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous [b, s, h, d] tensor")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    b, sq, h, d = q.shape
    if k.shape != v.shape or k.shape[0] != b or k.shape[2] != h or k.shape[3] != d:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    dt = _dtype_code(q)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or out.device.type != "cpu":
        raise ValueError("out must be a contiguous CPU tensor like q")
    if lse is None:
        lse = torch.empty((b, h, sq), dtype=torch.float32, pin_memory=True)
    elif (tuple(lse.shape) != (b, h, sq) or lse.dtype != torch.float32 or not lse.is_contiguous()
          or lse.device.type != "cpu"):
        raise ValueError("lse must be a contiguous float32 CPU tensor [b, h, sq]")
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    lib = load_library()
    with torch.cuda.device(device):
        st = _stream(device, stream)
        rc = lib.attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                               lse.data_ptr(), b, sq, k.shape[1], h, d, scale, dt, 1 if causal else 0, st)
        if rc != ATTN_OK:
            raise AttnError(rc, "attn_fwd_host")
        if sync:
            (torch.cuda.current_stream(device) if stream is None else stream).synchronize()
    return out, lse


def attn_decode_splitkv(q, k, v, scale: float | None = None, num_splits: int = 0, out=None,
                        lse=None, stream=None, causal: bool = False):
    """Split-KV decode: same result as attn_fwd, computed by splitting the
    keys into ``num_splits`` ranges (0 = heuristic) and reducing the
    per-split (O_i, LSE_i) with the log-sum-exp combine."""
    b, sq, sk, h, d, dt, idx = _check(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out, lse = _outputs(q, out, lse, b, h, sq, idx)
    lib = _lib or load_library()
    fn = lib.attn_decode_splitkv_causal if causal else lib.attn_decode_splitkv_ex
    rc = _call(fn, idx, stream, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
               lse.data_ptr(), b, sq, sk, h, d, scale, int(num_splits), dt)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_splitkv")
    return out, lse


def attn_decode_paged(q, k_pages, v_pages, block_table, seqlens_k, scale: float | None = None,
                      num_splits: int = 0, out=None, lse=None, stream=None, causal: bool = False):
    """Split-KV decode of the new rows of each sequence from a paged KV cache.

    q: [b, sq, h, d] (sq new rows per sequence); k_pages, v_pages:
    [num_pages, page_size, h, d] (page_size a multiple of 16); block_table:
    int32 [b, max_pages] pool page of each logical page; seqlens_k: int32
    [b] keys per sequence. All CUDA tensors. ``causal``: the
    bottom-right-aligned mask against each sequence's own key count."""
    if not isinstance(q, torch.Tensor) or not q.is_cuda or q.dim() != 4:
        raise ValueError("q must be a CUDA tensor [b, sq, h, d]")
    for name, t in (("k_pages", k_pages), ("v_pages", v_pages)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor [num_pages, page_size, h, d]")
        if t.dtype != q.dtype or t.device != q.device:
            raise ValueError(f"{name} must match q's dtype and device")
    if k_pages.shape != v_pages.shape:
        raise ValueError("k_pages and v_pages must have the same shape")
    for name, t in (("block_table", block_table), ("seqlens_k", seqlens_k)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.int32 or not t.is_cuda \
                or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor on q's device")
    if not q.is_contiguous():
        raise ValueError("q must be contiguous")
    b, sq, h, d = q.shape
    num_pages, page_size = k_pages.shape[0], k_pages.shape[1]
    if k_pages.shape[2] != h or k_pages.shape[3] != d:
        raise ValueError("page pools must be [num_pages, page_size, h, d] with q's h and d")
    if block_table.dim() != 2 or block_table.shape[0] != b or tuple(seqlens_k.shape) != (b,):
        raise ValueError("block_table must be [b, max_pages] and seqlens_k [b]")
    dt = _dtype_code(q)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    idx = q.get_device()
    out, lse = _outputs(q, out, lse, b, h, sq, idx)
    lib = _lib or load_library()
    rc = _call(lib.attn_decode_paged_ex, idx, stream, q.data_ptr(), k_pages.data_ptr(),
               v_pages.data_ptr(), block_table.data_ptr(), seqlens_k.data_ptr(), out.data_ptr(),
               lse.data_ptr(), b, sq, h, d, num_pages, page_size, block_table.shape[1], scale,
               int(num_splits), 1 if causal else 0, dt)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_paged")
    return out, lse


def attn_bwd(q, k, v, o, lse, dout, scale: float | None = None, dq=None, dk=None, dv=None,
             stream=None, causal: bool = False):
    """Backward pass of attn_fwd: returns (dq, dk, dv).

    q, o, dout: [b, sq, h, d]; k, v: [b, sk, h, d] (fp16 or bf16, contiguous
    CUDA tensors); lse: fp32 [b, h, sq] from attn_fwd with the same
    ``causal`` (the bottom-right-aligned mask, attn_bwd_causal)."""
    b, sq, sk, h, d, dt, idx = _check(q, k, v)
    for name, t in (("o", o), ("dout", dout)):
        if not isinstance(t, torch.Tensor) or t.shape != q.shape or t.dtype != q.dtype \
                or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous tensor like q")
    if (tuple(lse.shape) != (b, h, sq) or lse.dtype != torch.float32 or not lse.is_contiguous()
            or lse.device != q.device):
        raise ValueError("lse must be a contiguous float32 tensor [b, h, sq]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t.shape != ref.shape or t.dtype != ref.dtype or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous tensor like {name[1]}")
    lib = _lib or load_library()
    fn = lib.attn_bwd_causal if causal else lib.attn_bwd
    rc = _call(fn, idx, stream, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
               lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
               b, sq, sk, h, d, scale, dt)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_bwd_causal" if causal else "attn_bwd")
    return dq, dk, dv


def attn_decode_splitkv_noalloc(q, k, v, out, lse, scale: float | None = None,
                                num_splits: int = 0, stream=None):
    """attn_decode_splitkv for callers that cannot allocate device memory:
    out and lse must be given, and the per-split partials live in a fixed
    array inside the library (calls that overlap on the GPU race on it).
    Its kernels' timeouts are read by attn_get_noalloc_status()."""
    b, sq, sk, h, d, dt, idx = _check(q, k, v)
    if out is None or lse is None:
        raise ValueError("out and lse must be given: this entry point allocates nothing")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    out, lse = _outputs(q, out, lse, b, h, sq, idx)
    lib = _lib or load_library()
    rc = _call(lib.attn_decode_splitkv_noalloc, idx, stream, q.data_ptr(), k.data_ptr(),
               v.data_ptr(), out.data_ptr(), lse.data_ptr(), b, sq, sk, h, d, scale,
               int(num_splits), dt)
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_decode_splitkv_noalloc")
    return out, lse


def attn_get_noalloc_status(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the status word of the
    no-allocation decode."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(device):
        return load_library().attn_get_noalloc_status(_stream(device, stream))


def attn_decode_num_splits(b: int, sq: int, sk: int, h: int, d: int) -> int:
    """Split count the heuristic picks on the current device."""
    return load_library().attn_decode_num_splits(b, sq, sk, h, d)


def attn_decode_num_splits_for_sms(b: int, sq: int, sk: int, h: int, d: int, num_sms: int) -> int:
    """Split count the heuristic picks for a device with ``num_sms`` SMs."""
    return load_library().attn_decode_num_splits_for_sms(b, sq, sk, h, d, num_sms)


def attn_get_device_status(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device status."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(device):
        return load_library().attn_get_device_status(_stream(device, stream))


def attn_last_timeout_site() -> int:
    return load_library().attn_last_timeout_site()


def attn_release_workspace() -> None:
    load_library().attn_release_workspace()


def attn_debug_set_flags(flags: int) -> None:
    load_library().attn_debug_set_flags(int(flags))


__all__ = [
    "AttnError", "attn_fwd", "attn_fwd_host", "attn_bwd", "attn_decode_splitkv",
    "attn_decode_paged", "attn_decode_splitkv_noalloc", "attn_get_noalloc_status",
    "attn_decode_num_splits",
    "attn_decode_num_splits_for_sms", "attn_get_device_status", "attn_last_timeout_site",
    "attn_release_workspace", "attn_debug_set_flags", "attn_status_string", "load_library",
]
