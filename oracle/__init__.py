"""fp64 CPU oracle for exact attention (ctypes binding over ``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may use this package; the CUDA library never
does, and this package never imports the CUDA library.

``attention`` follows the standard (unfused) attention of "Why FlashAttention
is fast" (section 2, item 4): it builds each score row in full, applies the
max-subtracted softmax, multiplies by V, and also returns the natural-log
log-sum-exp of each score row. ``combine`` is the split-KV reduce stated in
the flash-decoding issue ("where is flash decoding second stage (reduce)
code?"): LSE = log(sum exp(LSE_i)) with the max taken out first, and
O = sum exp(LSE_i - LSE) * O_i.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F64, F32, F16, BF16 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, OpenMP, -O2)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-std=c11", "-Wall", "-shared", "-fPIC",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            lib.oracle_attn.restype = i32
            lib.oracle_attn.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, dbl,
                                        i32, i32, i32, vp, i32, vp, vp]
            lib.oracle_combine.restype = i32
            lib.oracle_combine.argtypes = [vp, vp, i32, ctypes.c_int64, i32, vp, vp]
            lib.oracle_f16_to_f64.restype = dbl
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = dbl
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_num_threads.restype = i32
            _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def _as_raw(x):
    """Return (contiguous numpy buffer, dtype code) without rounding anything."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        if x.is_cuda:
            raise ValueError("the oracle takes host tensors only")
        x = x.contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), BF16
        if x.dtype == torch.float16:
            return x.view(torch.int16).numpy().view(np.uint16), F16
        if x.dtype == torch.float32:
            return x.numpy(), F32
        if x.dtype == torch.float64:
            return x.numpy(), F64
        raise TypeError(f"unsupported dtype {x.dtype}")
    a = np.ascontiguousarray(x)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.float16:
        return a.view(np.uint16), F16
    raise TypeError(f"unsupported dtype {a.dtype}")


def attention(q, k, v, scale: float, rows=None, key_range=None, causal=False):
    """Exact attention in fp64.

    q: [b, sq, h, d]; k, v: [b, sk, h, d] (torch CPU tensors or numpy arrays,
    fp64/fp32/fp16/bf16; all three the same dtype).
    rows: optional list of query rows to evaluate (default: all sq).
    key_range: optional (j0, j1); only keys j0 <= j < j1 take part.
    causal: bottom-right-aligned causal mask (not on the pages; the common
    reading): query row i sees key j only if j <= i + sk - sq. A row left
    with no key gives O = 0 and LSE = -inf.
    Returns (o [b, nrows, h, d], lse [b, h, nrows]) as float64 numpy arrays.
    """
    qa, dt = _as_raw(q)
    ka, dtk = _as_raw(k)
    va, dtv = _as_raw(v)
    if not (dt == dtk == dtv):
        raise TypeError("q, k, v must share a dtype")
    b, sq, h, d = qa.shape
    bk, sk, hk, dk = ka.shape
    if va.shape != ka.shape or (bk, hk, dk) != (b, h, d):
        raise ValueError("shape mismatch")
    j0, j1 = (0, sk) if key_range is None else key_range
    if rows is None:
        rows_arr, nrows, rows_ptr = None, sq, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        nrows = int(rows_arr.size)
        rows_ptr = rows_arr.ctypes.data
    o = np.empty((b, nrows, h, d), dtype=np.float64)
    lse = np.empty((b, h, nrows), dtype=np.float64)
    rc = _load().oracle_attn(qa.ctypes.data, ka.ctypes.data, va.ctypes.data, dt,
                             b, sq, sk, h, d, float(scale), int(j0), int(j1), int(bool(causal)),
                             rows_ptr, nrows, o.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_attn rejected its arguments")
    return o, lse


def combine(o_parts, lse_parts):
    """Split-KV reduce in fp64.

    o_parts: [nsplit, R, d]; lse_parts: [nsplit, R] (any consistent row order).
    Returns (o [R, d], lse [R]).
    """
    op = np.ascontiguousarray(o_parts, dtype=np.float64)
    lp = np.ascontiguousarray(lse_parts, dtype=np.float64)
    ns, R, d = op.shape
    if lp.shape != (ns, R):
        raise ValueError("shape mismatch")
    o = np.empty((R, d), dtype=np.float64)
    lse = np.empty((R,), dtype=np.float64)
    rc = _load().oracle_combine(op.ctypes.data, lp.ctypes.data, ns, R, d,
                                o.ctypes.data, lse.ctypes.data)
    if rc != 0:
        raise ValueError("oracle_combine rejected its arguments")
    return o, lse


def split_attention(q, k, v, scale: float, bounds, rows=None, causal=False):
    """Per-split (O_i, LSE_i) over the key ranges ``bounds`` = [(j0, j1), ...],
    combined by ``combine``. Returns (o [b, nrows, h, d], lse [b, h, nrows])."""
    parts_o, parts_l = [], []
    for (j0, j1) in bounds:
        o_i, l_i = attention(q, k, v, scale, rows=rows, key_range=(j0, j1), causal=causal)
        b, nr, h, d = o_i.shape
        # put both in (b, h, row) order for the reduce
        parts_o.append(o_i.transpose(0, 2, 1, 3).reshape(b * h * nr, d))
        parts_l.append(l_i.reshape(b * h * nr))
    o, lse = combine(np.stack(parts_o), np.stack(parts_l))
    o = o.reshape(b, h, nr, d).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(o), lse.reshape(b, h, nr)


def decode_f16(bits: int) -> float:
    return _load().oracle_f16_to_f64(bits)


def decode_bf16(bits: int) -> float:
    return _load().oracle_bf16_to_f64(bits)


def paged_attention(q, k_pages, v_pages, block_table, seqlens, scale: float, causal=False):
    """Exact attention of each sequence's query rows over its own keys, read
    through a page table (a paged KV cache; the pages only mention one, so
    the layout is the common one): key r of sequence i is row r % page_size
    of pool page block_table[i, r // page_size], and sequence i has
    seqlens[i] keys. The keys are gathered into one contiguous cache per
    sequence and passed to ``attention``; a sequence with no key gives O = 0
    and LSE = -inf.

    causal: the bottom-right-aligned mask of ``attention`` taken against the
    sequence's own key count: its sq query rows are the last sq positions of
    its seqlens[i] keys, so row r sees key j only if j <= r + seqlens[i] - sq.

    q: [b, sq, h, d]; k_pages, v_pages: [num_pages, page_size, h, d];
    block_table: [b, max_pages] ints; seqlens: [b] ints (CPU tensors or
    numpy arrays). Returns (o [b, sq, h, d], lse [b, h, sq]) fp64."""
    table = np.asarray(block_table)
    lens = np.asarray(seqlens)
    page_size = k_pages.shape[1]
    outs_o, outs_l = [], []
    for i in range(q.shape[0]):
        n = int(lens[i])
        npg = (n + page_size - 1) // page_size
        if n == 0:
            keys = [int(table[i, 0])]  # any one page; the key range below is empty
        else:
            keys = [int(table[i, p]) for p in range(npg)]
        kc = _stack_pages(k_pages, keys)
        vc = _stack_pages(v_pages, keys)
        if causal and n > 0:
            # the mask is relative to the sequence's own keys: cut the gathered
            # cache to exactly n keys
            o_i, l_i = attention(q[i:i + 1], kc[:, :n], vc[:, :n], scale, causal=True)
        else:
            o_i, l_i = attention(q[i:i + 1], kc, vc, scale, key_range=(0, n))
        outs_o.append(o_i)
        outs_l.append(l_i)
    return np.concatenate(outs_o, axis=0), np.concatenate(outs_l, axis=0)


def _stack_pages(pool, pages):
    """[1, len(pages) * page_size, h, d]: the listed pool pages in order."""
    if isinstance(pool, np.ndarray):
        return np.concatenate([pool[p] for p in pages], axis=0)[None]
    import torch

    return torch.cat([pool[p] for p in pages], dim=0).unsqueeze(0).contiguous()


def _f64(x):
    """fp64 copy of a host tensor or array (16-bit values widen exactly)."""
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        if x.is_cuda:
            raise ValueError("the oracle takes host tensors only")
        return x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def attention_backward(q, k, v, do, scale: float, causal=False):
    """Gradients of the exact attention of ``attention``, by the chain rule of
    its plain definition (the flash-attn timing issue times a backward pass;
    none of the pages writes one out). With S = scale * Q K^T, P = softmax(S)
    row by row, O = P V and the upstream gradient dO:
        dV = P^T dO,   dP = dO V^T,   D = rowsum(P * dP),   dS = P * (dP - D),
        dQ = scale * dS K,   dK = scale * dS^T Q.
    With ``causal`` the masked scores of ``attention`` (bottom-right aligned)
    have P = 0; a row that sees no key has P = 0 throughout.

    q, do: [b, sq, h, d]; k, v: [b, sk, h, d] (host tensors or arrays).
    Returns (dq, dk, dv) as fp64 numpy arrays of the input shapes."""
    Q, K, V, dO = (_f64(t) for t in (q, k, v, do))
    b, sq, h, d = Q.shape
    sk = K.shape[1]
    dq, dk, dv = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    visible = np.ones((sq, sk), dtype=bool)
    if causal:
        visible = np.arange(sk)[None, :] <= np.arange(sq)[:, None] + (sk - sq)
    for bb in range(b):
        for hh in range(h):
            Qh, Kh, Vh, dOh = Q[bb, :, hh], K[bb, :, hh], V[bb, :, hh], dO[bb, :, hh]
            S = np.where(visible, scale * (Qh @ Kh.T), -np.inf)
            P = np.zeros_like(S)
            seen = visible.any(axis=1)
            Ss = S[seen]
            E = np.exp(Ss - Ss.max(axis=1, keepdims=True))
            P[seen] = E / E.sum(axis=1, keepdims=True)
            dP = dOh @ Vh.T
            D = (P * dP).sum(axis=1, keepdims=True)
            dS = P * (dP - D)
            dq[bb, :, hh] = scale * (dS @ Kh)
            dk[bb, :, hh] = scale * (dS.T @ Qh)
            dv[bb, :, hh] = P.T @ dOh
    return dq, dk, dv
