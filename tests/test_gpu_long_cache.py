"""Parity at the long-cache points of the decode sweep, at full size.

The decode sweep's bandwidth figures at long caches (20 query heads over 20 or 4 KV
heads, fp16) come from these shapes; here the same launch configuration is checked
against the fp64 oracle. The caches (up to 2.7 GB) are drawn on the device with a
seeded generator; the rows under test are copied back and the oracle recomputes every
output of those rows (all query heads) from the same bits. The sampled rows always
include the first and the last row and the rows with the shortest and the longest
length; lengths are ragged, with one row at the full capacity (the bench's length).
Both the plain launch and the launch with PDL and early K/V staging are checked.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attn_close, host16, new_err, require_gpu
from workloads import gen_cache_device, gen_queries, make_rng

pytestmark = pytest.mark.gpu
D = 64


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


SHAPES = [  # (batch, q heads, kv heads, capacity)
    (64, 20, 20, 8192),
    (64, 20, 4, 8192),
    (16, 20, 20, 2048),
    (16, 20, 4, 2048),
]


def _sample_rows(rng, lens, n_extra=4):
    B = len(lens)
    rows = {0, B - 1, int(np.argmin(lens)), int(np.argmax(lens))}
    rows |= set(int(r) for r in rng.choice(B, size=min(B, n_extra), replace=False))
    return sorted(rows)


@pytest.mark.parametrize("shape", SHAPES, ids=[f"B{b}-{hq}/{hk}-L{L}" for b, hq, hk, L in SHAPES])
def test_long_cache_decode_sampled_rows(shape):
    import kv_cached_decode_gb300 as kvd

    B, Hq, Hkv, L = shape
    dtype = "f16"
    seed = 31000 + B * 10 + Hkv + L
    rng = make_rng(seed)
    lens = rng.integers(L // 2, L + 1, size=B).astype(np.int32)
    lens[rng.integers(0, B)] = L  # one row at the full capacity
    K, V = gen_cache_device(seed, B, Hkv, L, D, dtype, 0.125)
    q = gen_queries(rng, B, Hq, 1, D, dtype, 0.125)
    qd = torch.from_numpy(q.view(np.int16)).view(torch.float16).cuda()
    lens_d = torch.from_numpy(lens).cuda()
    cache = kvd.make_cache(K, V)
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_DECODE_ATTN, B, Hq, Hkv, 1, 1, L))
    outs = {}
    for flags in (0, kvd.KVD_FLAG_PDL | kvd.KVD_FLAG_EARLY_KV):
        out = torch.full_like(qd, 3.0)
        err = new_err()
        kvd.kvd_decode_attn(qd, cache, out, ws, lens=lens_d, flags=flags, dev_err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        outs[flags] = host16(out)
    rows = _sample_rows(rng, lens)
    idx = torch.tensor(rows, device="cuda")
    Ks = host16(K.index_select(0, idx))
    Vs = host16(V.index_select(0, idx))
    want, errs = oracle.attention(q[rows], Ks, Vs, dtype, lens=lens[rows])
    assert not errs
    for flags, got in outs.items():
        assert_attn_close(got[rows], want, dtype, f"rows {rows}, flags {flags}")
    # the two launch forms run the same plan and merge order: identical bits everywhere
    assert np.array_equal(outs[0], outs[kvd.KVD_FLAG_PDL | kvd.KVD_FLAG_EARLY_KV])
