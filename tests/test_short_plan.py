"""The short forward kernel's launch plan, checked on the host (no GPU).

attn_debug_short_plan returns the plan attn_fwd would launch the short
kernel with: how the CTA's 512 TMEM columns are cut into slots (S, then P
in S's first half, then O) and how its shared memory is cut into query
stages and, with heads in groups of four, a K/V ring. A plan that overflowed
either would corrupt or fault on the GPU, so every shape class the kernel
takes is checked here: key counts on both sides of each 32-key chunk edge
up to 256, one to many query rows, head counts with and without groups of
four, every head dim, grouping allowed or not.
"""
import ctypes
import itertools

import pytest

SKS = [1, 5, 31, 32, 33, 64, 100, 128, 150, 160, 161, 192, 200, 224, 255, 256]
TMEM_COLS = 512


def _plan(lib, sq, sk, h, d, grouped_ok, out=True):
    fn = lib.attn_debug_short_plan
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int)]
    buf = (ctypes.c_int * 12)(*([-7] * 12))
    ok = fn(sq, sk, h, d, grouped_ok, buf if out else None)
    return ok, list(buf)


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("grouped_ok", [0, 1])
def test_plans_fit_tmem_and_shared_memory(exattn_lib, d, grouped_ok):
    for sk, sq, h in itertools.product(SKS, [1, 20, 150, 1000], [1, 3, 4, 8, 16]):
        ok, p = _plan(exattn_lib, sq, sk, h, d, grouped_ok)
        assert ok == 1, (sq, sk, h, d)
        n, o_off, w, nslot, kv_bytes, stage_bytes, nstage, grouped, nblk, nkv, used, avail = p
        assert n == (sk + 31) // 32 * 32 <= 256
        # heads are grouped exactly when allowed, at d = 16 with heads in fours
        assert grouped == int(bool(grouped_ok) and d == 16 and h % 4 == 0)
        # TMEM: whole 32-column slots, all within the 512 columns
        assert w % 32 == 0 and 1 <= nslot <= 3 and nslot * w <= TMEM_COLS
        # S takes the first N columns, P (16-bit pairs) the first N / 2, and
        # O (the four heads' 64 columns when grouped) lies past P in the slot
        o_cols = 64 if grouped else d
        assert n <= w and o_off >= n // 2 and o_off + o_cols <= w
        # shared memory: the tiles fit, and every tile starts on a 1024-byte
        # boundary (the widest swizzle pattern)
        assert 0 < used <= avail
        assert stage_bytes % 1024 == 0 and kv_bytes % 1024 == 0
        # the P V issuer runs up to nslot - 1 items behind QK^T, so the ring
        # holds at least one item per slot
        assert nstage >= nslot >= 1
        if grouped:
            assert nblk == (sq + 31) // 32 and nkv in (2, 3)
            assert stage_bytes == 32 * 128 + 128 * 128  # staging block + diagonal tile
            assert kv_bytes == n * 128                  # N keys of four heads' 16 columns
            assert used == nstage * stage_bytes + nkv * 2 * kv_bytes
        else:
            assert nblk == 0 and nkv == 0
            assert kv_bytes == n * d * 2
            assert stage_bytes == 128 * d * 2 + 2 * kv_bytes  # Q tile, K, V
            assert used == nstage * stage_bytes


def test_items_in_flight_for_the_small_head_problem(exattn_lib):
    """b512 s150 h16 d16 (heads in fours): N = 160, three slots of 160
    columns, O at column 96, the group's K and V in a ring of three."""
    ok, p = _plan(exattn_lib, 150, 150, 16, 16, 1)
    assert ok == 1
    n, o_off, w, nslot, kv_bytes, stage_bytes, nstage, grouped, nblk, nkv, used, avail = p
    assert (n, o_off, w, nslot, grouped, nblk, nkv) == (160, 96, 160, 3, 1, 5, 3)


@pytest.mark.parametrize("sq,sk,h,d", [(150, 257, 16, 16), (150, 150, 16, 128), (150, 150, 16, 8),
                                       (0, 150, 16, 16), (150, 0, 16, 16), (150, 150, 0, 16)])
def test_shapes_the_short_kernel_does_not_take(exattn_lib, sq, sk, h, d):
    ok, p = _plan(exattn_lib, sq, sk, h, d, 1)
    assert ok == 0 and p == [-7] * 12


def test_no_output_buffer(exattn_lib):
    ok, _ = _plan(exattn_lib, 150, 150, 16, 16, 1, out=False)
    assert ok == 0
