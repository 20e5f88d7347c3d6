"""kvd_decode_attn_noalloc: decode attention for callers that cannot allocate.

Callers such as plugin or custom-op interfaces that only hand over input and output
pointers, or servers that reserve all device memory at start-up, cannot give the
library a workspace. This entry point merges split results in a scratch buffer built
into the library instead. The test calls it through the C ABI twice in a row and
checks both outputs against the workspace entry point's output (and the fp64 oracle)
with the attention tolerance used everywhere else: max-abs 1e-2, rel-Frobenius 5e-3.

Kept in a file of its own that pytest collects last; it must pass alone in a fresh
process and after every other test.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attn_close, attn_errors, dev16, dev_i32, host16, new_err, require_gpu
from workloads import gen_cache, gen_queries, make_rng

pytestmark = pytest.mark.gpu
D = 64


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


# (dtype, batch, q heads, kv heads, capacity, lengths or None, fixed length)
CASES = [
    # two (row, head) units over 32768 positions: 8 clusters of 16 splits per unit, the
    # clusters' partials merged in the scratch buffer
    ("f16", 1, 2, 2, 32768, [32000], 0),
    # ragged GQA rows: merged inside thread-block clusters, scratch counters unused
    ("bf16", 4, 9, 3, 700, [700, 1, 333, 64], 0),
    # cross attention over 1500 frames with beam rows sharing each window's K/V
    ("f16", 6, 4, 4, 1500, None, 1500),
]


@pytest.mark.parametrize("case", CASES, ids=["workspace-merge", "gqa-ragged", "beam-cross"])
def test_noalloc_matches_workspace_entry_point_twice(case):
    import kv_cached_decode_gb300 as kvd

    dtype, B, Hq, Hkv, cap, lens, fixed = case
    rpk = 3 if fixed else 1
    rng = make_rng(9000 + B + cap)
    K, V = gen_cache(rng, B // rpk, Hkv, cap, D, dtype, 0.125,
                     lens=lens if lens is not None else [fixed] * (B // rpk))
    q = gen_queries(rng, B, Hq, 1, D, dtype, 0.125)
    lens_np = None if lens is None else np.array(lens, np.int32)
    want, _ = oracle.attention(q, K, V, dtype, lens=lens_np, fixed_len=fixed, rows_per_kv=rpk)

    Kd, Vd, qd = dev16(K, dtype), dev16(V, dtype), dev16(q, dtype)
    cache = kvd.make_cache(Kd, Vd)
    lens_d = None if lens is None else dev_i32(lens)
    ref = torch.empty_like(qd)
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_DECODE_ATTN, B, Hq, Hkv, rpk, 1,
                                                  cap if lens is not None else fixed))
    kvd.kvd_decode_attn(qd, cache, ref, ws, lens=lens_d, fixed_len=fixed, rows_per_kv=rpk)
    err = new_err()
    outs = []
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        o = torch.full_like(qd, 3.0)
        kvd.kvd_decode_attn_noalloc(qd, cache, o, lens=lens_d, fixed_len=fixed,
                                    rows_per_kv=rpk, dev_err=err)
        outs.append(o)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref_bits = host16(ref)
    for o in outs:
        got = host16(o)
        max_abs, rel = attn_errors(got, ref_bits.view(np.float16).astype(np.float64)
                                   if dtype == "f16" else
                                   (ref_bits.astype(np.uint32) << 16).view(np.float32)
                                   .astype(np.float64), dtype)
        assert max_abs <= 1e-2 and rel <= 5e-3, (max_abs, rel)
        assert_attn_close(got, want, dtype, "noalloc vs oracle")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    import kv_cached_decode_gb300 as kvd

    # 8 KV heads x 16 query heads each over 32768 positions: plain splits merged through
    # the scratch (at most about 2 clusters per unit fit at once), 8 units x 30 or more
    # splits x 16 query vectors: over 1 MiB of partials, more than the built-in 512 KiB.
    K = torch.zeros(1, 8, 32768, D, dtype=torch.float16, device="cuda")
    q = torch.zeros(1, 128, 1, D, dtype=torch.float16, device="cuda")
    out = torch.full_like(q, 5.0)
    with pytest.raises(kvd.KvdError) as ei:
        kvd.kvd_decode_attn_noalloc(q, kvd.make_cache(K, K), out, fixed_len=32768)
    assert ei.value.status == 3  # KVD_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 5.0)


def test_noalloc_recovers_from_counters_left_non_zero():
    """A call that stopped early (a timed-out wait) can leave the built-in scratch's
    arrival counters non-zero. The counters are overwritten here from the host (no fault,
    no stalled kernel), then the next call must still merge from zero: its output equals
    the workspace entry point's bit for bit (same plan, same merge order)."""
    import kv_cached_decode_gb300 as kvd

    dtype, B, Hq, Hkv, cap, lens, fixed = CASES[0]  # merges through the scratch
    rng = make_rng(9100)
    K, V = gen_cache(rng, B, Hkv, cap, D, dtype, 0.125, lens=lens)
    q = gen_queries(rng, B, Hq, 1, D, dtype, 0.125)
    Kd, Vd, qd = dev16(K, dtype), dev16(V, dtype), dev16(q, dtype)
    cache = kvd.make_cache(Kd, Vd)
    lens_d = dev_i32(lens)
    ref = torch.empty_like(qd)
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_DECODE_ATTN, B, Hq, Hkv, 1, 1, cap))
    kvd.kvd_decode_attn(qd, cache, ref, ws, lens=lens_d)
    err = new_err()
    for fill in (0x01, 0x7F):
        kvd.kvd_noalloc_test_fill_counters(fill)
        o = torch.full_like(qd, 3.0)
        kvd.kvd_decode_attn_noalloc(qd, cache, o, lens=lens_d, dev_err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert np.array_equal(host16(o), host16(ref)), f"fill {fill:#x}"


def test_noalloc_after_a_call_that_gave_up():
    """A call that really stopped early: with KVD_FLAG_TEST_STALL the last split of the
    unit gives up after a bounded wait (KVD_ERR_TIMEOUT, output unwritten), leaving the
    built-in scratch's arrival counter part-way. The next call, with nothing re-zeroed by
    the caller, must still equal the workspace entry point bit for bit."""
    import kv_cached_decode_gb300 as kvd

    dtype, B, Hq, Hkv, cap, _, fixed = CASES[0]  # merges through the scratch
    lens = [cap]  # a full row: the last split has tiles, so its first stage is the one stalled
    rng = make_rng(9200)
    K, V = gen_cache(rng, B, Hkv, cap, D, dtype, 0.125, lens=lens)
    q = gen_queries(rng, B, Hq, 1, D, dtype, 0.125)
    Kd, Vd, qd = dev16(K, dtype), dev16(V, dtype), dev16(q, dtype)
    cache = kvd.make_cache(Kd, Vd)
    lens_d = dev_i32(lens)
    ref = torch.empty_like(qd)
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_DECODE_ATTN, B, Hq, Hkv, 1, 1, cap))
    kvd.kvd_decode_attn(qd, cache, ref, ws, lens=lens_d)
    stalled = torch.full_like(qd, 3.0)
    err = new_err()
    kvd.kvd_decode_attn_noalloc(qd, cache, stalled, lens=lens_d, dev_err=err,
                                flags=kvd.KVD_FLAG_TEST_STALL)
    torch.cuda.synchronize()
    assert err.item() == 20  # KVD_ERR_TIMEOUT
    assert torch.all(stalled == 3.0)
    o = torch.full_like(qd, 3.0)
    err2 = new_err()
    kvd.kvd_decode_attn_noalloc(qd, cache, o, lens=lens_d, dev_err=err2)
    torch.cuda.synchronize()
    assert err2.item() == 0
    assert np.array_equal(host16(o), host16(ref))
