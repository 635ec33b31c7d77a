"""Host-side checks of the C ABI; none of these launches a kernel or needs a GPU.

* the library builds for sm_103a, loads, and exports every function that
  include/exattn.h declares;
* argument validation returns its status before touching any pointer;
* the split heuristic (pure host arithmetic) follows the rule of the
  flash-decoding issue: no split once the work units cover the SMs (b=8,
  h=48 gives 384 units: one split), more splits otherwise. A unit is
  b*h*ceil(sq/rows) for one query row (CUDA-core kernel) and 256 query rows
  of a (batch, head) for several (tensor-core kernel).
"""
import ctypes
import re

import pytest

import exact_attention_65_gb300 as ea

ALIGNED = 0x10000  # never dereferenced: validation fails before any use


def declared_functions():
    text = open(ea.HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(exattn_lib):
    names = declared_functions()
    assert "attn_fwd" in names and "attn_decode_splitkv" in names
    for name in names:
        assert hasattr(exattn_lib, name), f"{name} is declared in exattn.h but not exported"


def test_version_and_status_strings(exattn_lib):
    assert ea.load_library().attn_version() >= 100
    seen = set()
    for code in range(6):
        s = ea.attn_status_string(code)
        assert s and s not in seen
        seen.add(s)
    assert ea.attn_status_string(99) == "unknown status"


def _fwd(lib, q=ALIGNED, k=ALIGNED, v=ALIGNED, o=ALIGNED, lse=ALIGNED, b=1, sq=8, sk=8, h=1, d=64,
         scale=0.125, dtype=ea.ATTN_BF16):
    return lib.attn_fwd(q, k, v, o, lse, b, sq, sk, h, d, scale, dtype, None)


def _dec(lib, q=ALIGNED, k=ALIGNED, v=ALIGNED, o=ALIGNED, lse=ALIGNED, b=1, sq=1, sk=8, h=1, d=64,
         scale=0.125, splits=0):
    return lib.attn_decode_splitkv(q, k, v, o, lse, b, sq, sk, h, d, scale, splits, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), ea.ATTN_ERR_INVALID_ARG),
    (dict(lse=None), ea.ATTN_ERR_INVALID_ARG),
    (dict(k=ALIGNED + 8), ea.ATTN_ERR_INVALID_ARG),      # not 16-byte aligned
    (dict(lse=ALIGNED + 2), ea.ATTN_ERR_INVALID_ARG),    # not 4-byte aligned
    (dict(b=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(sq=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(sk=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(h=-1), ea.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), ea.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), ea.ATTN_ERR_INVALID_ARG),
    (dict(dtype=7), ea.ATTN_ERR_INVALID_ARG),
    (dict(d=48), ea.ATTN_ERR_UNSUPPORTED),
    (dict(d=256), ea.ATTN_ERR_UNSUPPORTED),
    (dict(d=8), ea.ATTN_ERR_UNSUPPORTED),
    (dict(b=70000), ea.ATTN_ERR_UNSUPPORTED),
])
def test_fwd_validation(exattn_lib, kw, expect):
    assert _fwd(exattn_lib, **kw) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(q=None), ea.ATTN_ERR_INVALID_ARG),
    (dict(o=ALIGNED + 8), ea.ATTN_ERR_INVALID_ARG),
    (dict(sq=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), ea.ATTN_ERR_INVALID_ARG),
    (dict(d=96), ea.ATTN_ERR_UNSUPPORTED),
])
def test_fwd_host_validation(exattn_lib, kw, expect):
    """The host-buffer forward checks its arguments before any CUDA call."""
    args = dict(q=ALIGNED, k=ALIGNED, v=ALIGNED, o=ALIGNED, lse=ALIGNED, b=1, sq=8, sk=8, h=1, d=64,
                scale=0.125)
    args.update(kw)
    a = args
    assert exattn_lib.attn_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["b"], a["sq"], a["sk"],
                                    a["h"], a["d"], a["scale"], ea.ATTN_BF16, 0, None) == expect


@pytest.mark.parametrize("kw,expect", [
    (dict(v=None), ea.ATTN_ERR_INVALID_ARG),
    (dict(o=ALIGNED + 4), ea.ATTN_ERR_INVALID_ARG),
    (dict(sk=0), ea.ATTN_ERR_INVALID_ARG),
    (dict(splits=-1), ea.ATTN_ERR_INVALID_ARG),
    (dict(d=96), ea.ATTN_ERR_UNSUPPORTED),
    (dict(b=70000), ea.ATTN_ERR_UNSUPPORTED),            # b beyond the grid limit
])
def test_decode_validation(exattn_lib, kw, expect):
    assert _dec(exattn_lib, **kw) == expect


def test_heuristic_follows_the_parallel_work_rule(exattn_lib):
    f = ea.attn_decode_num_splits_for_sms
    # b=8, h=48, sq=1: 384 units >= SMs, so no split (A100's 108 as in the
    # issue, and a GB300's SM count).
    for sms in (108, 132, 148, 152):
        assert f(8, 1, 8192, 48, 128, sms) == 1
    # b=1, h=16, sq=1: 16 units leave SMs idle, so split; as many CTAs as fit
    # one per SM.
    for sms in (148, 152):
        s = f(1, 1, 32768, 16, 128, sms)
        assert s == sms // 16
        assert 16 * s <= sms < 16 * (s + 1)
    # never more splits than key blocks (64 rows of d=128 per block)
    assert f(1, 1, 100, 1, 128, 148) == 2
    assert f(1, 1, 1, 1, 128, 148) == 1
    # sq > 1 runs on the tensor-core kernel: a unit is 256 query rows of one
    # (batch, head), a split at least one 128-key tile
    assert f(2, 10, 65536, 8, 128, 148) == 148 // (2 * 8)
    assert f(2, 300, 65536, 8, 128, 148) == 148 // (2 * 8 * 2)
    assert f(1, 10, 300, 16, 128, 152) == 3          # three key tiles
    # the flash-decoding issue's workload: b8, 48 heads, 1 to 10 new rows: no split
    for sq in range(1, 11):
        assert f(8, sq, 8192, 48, 128, 152) == 1
    # 100 units: two splits would need 200 CTAs, more than the SMs, so one
    assert f(1, 1, 65536, 100, 128, 148) == 1
    # more work units than SMs at any sq
    assert f(64, 16, 4096, 32, 64, 148) == 1
    # invalid sizes
    assert f(0, 1, 10, 1, 128, 148) == 0
    assert f(1, 1, 10, 1, 100, 148) == 0
    assert f(1, 1, 10, 1, 128, 0) == 0


def test_heuristic_monotone_in_work(exattn_lib):
    f = ea.attn_decode_num_splits_for_sms
    prev = None
    for h in (1, 2, 4, 8, 16, 32, 64, 128, 256):
        s = f(1, 1, 1 << 20, h, 128, 148)
        assert s >= 1
        if prev is not None:
            assert s <= prev
        prev = s
    assert prev == 1


def test_product_path_has_no_fallback(tmp_path, monkeypatch):
    """Without the built library the binding refuses to run."""
    monkeypatch.setattr(ea, "_lib", None)
    monkeypatch.setattr(ea, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        ea.load_library()


def test_binding_rejects_host_tensors():
    import torch

    q = torch.zeros(1, 4, 1, 16, dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ea.attn_fwd(q, q, q)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ea.attn_decode_splitkv(q, q, q)
