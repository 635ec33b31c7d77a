"""Negative softmax scales on every kernel that computes S on the tensor core.

With scale < 0 the largest scaled score of a row is scale times its
smallest raw score. The kernels do not track that minimum: their S MMAs
negate Q when the scale is negative, so the scores reach the softmax
already multiplied by the sign, and it works with |scale| (negation is
exact, so the products are the same). Each case runs one compiled form
against the fp64 oracle, at scale -s and +s. Q is scaled up so that the
scaled scores have a standard deviation of about 3 (a spread of about 20
units per row): a row max taken on the wrong side would then overflow or
lose the row. Forms covered: the plain forward and the causal
forward, with ragged key tiles; the one-live-tile form (plain and causal);
the key-range form of several-row split decode; the short kernel, one head
per item (d = 32) and heads in groups of four (d = 16); and the CUDA-core
one-row decode, which folds the scale into q. Tolerance as everywhere:
max |O - O_ref| <= 2e-2, max |LSE - LSE_ref| <= 1e-3 (on rows that see a key).
"""
import pytest
import torch

import workloads
from parity import compare, compare_masked

pytestmark = pytest.mark.gpu


def _inputs(b, sq, sk, h, d, dtype, seed, q_gain):
    q, k, v = workloads.make_qkv(b, sq, sk, h, d, dtype, seed=seed)
    q = (q.float() * q_gain).to(dtype)
    return q, k, v


CASES = [
    # name, (b, sq, sk, h, d), dtype, scale magnitude, q gain, causal, path
    ("plain", (1, 300, 600, 2, 128), torch.bfloat16, 0.09, 3.0, False, "fwd"),
    ("causal", (1, 300, 600, 2, 128), torch.bfloat16, 0.09, 3.0, True, "fwd"),
    ("one_tile", (2, 64, 1000, 2, 64), torch.float16, 0.125, 3.0, False, "fwd"),
    ("one_tile_causal", (2, 64, 1000, 2, 64), torch.float16, 0.125, 3.0, True, "fwd"),
    ("key_ranges", (2, 10, 3000, 3, 128), torch.bfloat16, 0.09, 3.0, False, "split4"),
    ("key_ranges_causal", (2, 10, 3000, 3, 128), torch.bfloat16, 0.09, 3.0, True, "split4"),
    ("short", (2, 150, 150, 3, 32), torch.float16, 0.18, 3.0, False, "fwd"),
    ("short_grouped", (48, 150, 150, 4, 16), torch.float16, 0.25, 3.0, False, "fwd"),
    ("short_grouped_bf16", (48, 97, 37, 4, 16), torch.bfloat16, 0.25, 3.0, False, "fwd"),
    ("one_row", (2, 1, 5000, 4, 128), torch.bfloat16, 0.09, 3.0, False, "split3"),
]


@pytest.mark.parametrize("sign", [-1.0, 1.0])
@pytest.mark.parametrize("name,shape,dtype,mag,gain,causal,path", CASES, ids=[c[0] for c in CASES])
def test_scale_sign(gpu, oracle_mod, sign, name, shape, dtype, mag, gain, causal, path):
    b, sq, sk, h, d = shape
    q, k, v = _inputs(b, sq, sk, h, d, dtype, seed=900 + sq + sk, q_gain=gain)
    scale = sign * mag
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    if path == "fwd":
        o, lse = gpu.attn_fwd(qd, kd, vd, scale=scale, causal=causal)
    else:
        splits = int(path[len("split"):])
        o, lse = gpu.attn_decode_splitkv(qd, kd, vd, scale=scale, num_splits=splits, causal=causal)
    assert gpu.attn_get_device_status() == gpu.ATTN_OK
    o_ref, lse_ref = oracle_mod.attention(q, k, v, scale, causal=causal)
    if causal:
        compare_masked(o, lse, o_ref, lse_ref)
    else:
        compare(o, lse, o_ref, lse_ref)
