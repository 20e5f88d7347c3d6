"""The attention kernels' bounded-wait failure path, driven on the GPU without a fault.

KVD_FLAG_TEST_STALL makes the first stage of the last split of every (row, KV head)
unit expect more bytes than its copies bring, so that split's tile waits run out after
about one second. The call must then report KVD_ERR_TIMEOUT, leave the output
unwritten, and leave the context and stream usable: the next normal call on the same
stream matches the fp64 oracle. Every
merge path is covered: one split per unit, the cluster merge (the split that gives up
is a non-first CTA, which sends nothing, so the first CTA's bounded wait for the
partials runs out and it writes no output), several clusters per unit merged through the
workspace (the stalled cluster's first CTA gives up, so the unit's last arrival never
comes), and plain splits merged through the workspace. After a workspace merge the
unit's arrival counter is left non-zero and the workspace is re-zeroed, as the header
says. Each stall costs a few seconds of waiting.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attn_close, dev16, dev_i32, host16, new_err, require_gpu
from workloads import gen_cache, gen_queries, make_rng

pytestmark = pytest.mark.gpu
D = 64
TIMEOUT = 20  # KVD_ERR_TIMEOUT


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


# (name, dtype, batch, q heads, kv heads, length, qlen) -- fixed lengths, so the last
# split of every unit has tiles to wait for
CASES = [
    ("one-split", "f16", 1, 2, 2, 64, 1),
    ("cluster-tensor-cores", "f16", 1, 20, 20, 1500, 1),
    ("cluster-cuda-cores", "bf16", 1, 4, 4, 4096, 1),
    ("cluster-verify-block", "f16", 1, 20, 20, 1500, 5),
    # 1 unit over 32768 positions: 8 clusters of 16 splits, merged through the workspace
    ("clusters-per-unit", "f16", 1, 1, 1, 32768, 1),
    # 8 GQA units over 32768 positions: plain splits merged through the workspace
    ("workspace-merge-plain", "f16", 2, 20, 4, 32768, 1),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_attention_wait_that_runs_out_reports_and_leaves_stream_usable(case):
    import kv_cached_decode_gb300 as kvd

    _, dtype, B, Hq, Hkv, L, qlen = case
    rng = make_rng(7100 + L + qlen)
    K, V = gen_cache(rng, B, Hkv, L, D, dtype, 0.125)
    q = gen_queries(rng, B, Hq, qlen, D, dtype, 0.125)
    want, _ = oracle.attention(q, K, V, dtype, fixed_len=L)
    Kd, Vd, qd = dev16(K, dtype), dev16(V, dtype), dev16(q, dtype)
    cache = kvd.make_cache(Kd, Vd)
    op = kvd.KVD_OP_DECODE_ATTN if qlen == 1 else kvd.KVD_OP_VERIFY_ATTN
    ws = kvd.new_workspace(kvd.kvd_workspace_size(op, B, Hq, Hkv, 1, qlen, L))

    def call(out, flags, err):
        if qlen == 1:
            kvd.kvd_decode_attn(qd, cache, out, ws, fixed_len=L, flags=flags, dev_err=err)
        else:
            kvd.kvd_verify_attn(qd, cache, out, ws, fixed_len=L, causal=False, flags=flags,
                                dev_err=err)

    out = torch.full_like(qd, 3.0)
    err = new_err()
    call(out, kvd.KVD_FLAG_TEST_STALL, err)
    torch.cuda.synchronize()
    assert err.item() == TIMEOUT
    assert torch.all(out == 3.0), "a unit whose split gave up wrote an output"
    # the workspace merge leaves the stalled unit's counter non-zero: re-zero it
    ws.zero_()
    out2 = torch.full_like(qd, 3.0)
    err2 = new_err()
    call(out2, 0, err2)
    torch.cuda.synchronize()
    assert err2.item() == 0
    assert_attn_close(host16(out2), want, dtype, "after a timeout")


def test_attention_timeout_with_pdl_chain_then_normal_chain():
    """The stall inside a chain of PDL launches over the same stream: the timed-out
    launch and the one after it both finish; a following normal chain matches the
    oracle (the dependent launch's wait is released by the stalled grid's exit)."""
    import kv_cached_decode_gb300 as kvd

    dtype, B, H, L = "f16", 1, 20, 1500
    rng = make_rng(7200)
    K, V = gen_cache(rng, B, H, L, D, dtype, 0.125)
    q = gen_queries(rng, B, H, 1, D, dtype, 0.125)
    want, _ = oracle.attention(q, K, V, dtype, fixed_len=L)
    Kd, Vd, qd = dev16(K, dtype), dev16(V, dtype), dev16(q, dtype)
    cache = kvd.make_cache(Kd, Vd)
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_DECODE_ATTN, B, H, H, 1, 1, L))
    pdl = kvd.KVD_FLAG_PDL | kvd.KVD_FLAG_EARLY_KV
    outs = [torch.full_like(qd, 3.0) for _ in range(3)]
    errs = [new_err() for _ in range(3)]
    kvd.kvd_decode_attn(qd, cache, outs[0], ws, fixed_len=L, flags=pdl, dev_err=errs[0])
    kvd.kvd_decode_attn(qd, cache, outs[1], ws, fixed_len=L, flags=pdl | kvd.KVD_FLAG_TEST_STALL,
                        dev_err=errs[1])
    kvd.kvd_decode_attn(qd, cache, outs[2], ws, fixed_len=L, flags=pdl, dev_err=errs[2])
    torch.cuda.synchronize()
    assert [e.item() for e in errs] == [0, TIMEOUT, 0]
    assert torch.all(outs[1] == 3.0)
    for i in (0, 2):
        assert_attn_close(host16(outs[i]), want, dtype, f"launch {i} of the chain")
    assert np.array_equal(host16(outs[0]), host16(outs[2]))
