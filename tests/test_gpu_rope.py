"""Rotary encoding on the GPU (kvd_rope) against the fp64 oracle.

Each rotated value must lie within one unit in the last place of the storage type of
the oracle's value (plus 2e-4 of the pair's norm for the fp32 angle and sin/cos). End
to end, a GQA decode step whose queries and new keys are rotated at their absolute
positions must match the oracle's rotation (rounded to the storage type) followed by
its append and attention, within the attention tolerance.
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attn_close, dev16, dev_i32, host16, new_err, require_gpu
from workloads import gen_cache, gen_new_kv, gen_queries, make_rng

pytestmark = pytest.mark.gpu
D = 64


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _to_f64(bits, dtype):
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _round_bits(x, dtype):
    """float64 -> fp16/bf16 bits, round to nearest even (through float32 for bf16)."""
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    f = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    r = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def _ulp(y, dtype):
    mant = 10 if dtype == "f16" else 7
    e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -14)))
    return 2.0 ** (e - mant)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_rope_matches_the_oracle(dtype):
    import kv_cached_decode_gb300 as kvd

    rng = make_rng(900)
    q = gen_queries(rng, 3, 9, 5, D, dtype, 1.0)
    k = gen_queries(rng, 3, 3, 5, D, dtype, 1.0)
    pos0 = np.array([0, 1000, 2047], np.int32)
    qd, kd = dev16(q, dtype), dev16(k, dtype)
    kvd.kvd_rope(qd, kd, dev_i32(pos0))
    torch.cuda.synchronize()
    for x, xd in ((q, qd), (k, kd)):
        want = oracle.rope(x, dtype, pos0)
        got = _to_f64(host16(xd), dtype)
        xf = _to_f64(x, dtype)
        pair = np.sqrt(xf[..., :32] ** 2 + xf[..., 32:] ** 2)
        pair = np.concatenate([pair, pair], axis=-1)
        assert np.all(np.abs(got - want) <= _ulp(want, dtype) + 2e-4 * pair)
    # position 0 leaves the first row's first token unchanged
    assert np.array_equal(host16(qd)[0, :, 0], q[0, :, 0])


def test_rope_then_gqa_decode_step():
    import kv_cached_decode_gb300 as kvd

    dtype, B, Hq, Hkv, cap = "bf16", 4, 9, 3, 1100
    rng = make_rng(901)
    lens = np.array([300, 1, 1000, 64], np.int32)
    K, V = gen_cache(rng, B, Hkv, cap, D, dtype, 0.125, lens=lens)
    kn, vn = gen_new_kv(rng, B, Hkv, 1, D, dtype, 0.125)
    q = gen_queries(rng, B, Hq, 1, D, dtype, 0.125)
    # oracle: rotate q and the new key at position lens[b], round, append, attend
    q_r = _round_bits(oracle.rope(q, dtype, lens), dtype)
    kn_r = _round_bits(oracle.rope(kn, dtype, lens), dtype)
    Kw, Vw = K.copy(), V.copy()
    lens_w, err = oracle.kv_append(Kw, Vw, kn_r, vn, lens, dtype)
    want, _ = oracle.attention(q_r, Kw, Vw, dtype, lens=lens_w)
    # GPU: rope in place, then decode with the fused append
    qd, knd, vnd = dev16(q, dtype), dev16(kn, dtype), dev16(vn, dtype)
    Kd, Vd = dev16(K, dtype), dev16(V, dtype)
    lens_d = dev_i32(lens)
    lens_out = torch.zeros_like(lens_d)
    out = torch.empty_like(qd)
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_DECODE_ATTN, B, Hq, Hkv, 1, 1, cap))
    e = new_err()
    kvd.kvd_rope(qd, knd, lens_d, flags=kvd.KVD_FLAG_PDL)
    kvd.kvd_decode_attn(qd, kvd.make_cache(Kd, Vd), out, ws, lens=lens_d, dev_err=e,
                        flags=kvd.KVD_FLAG_PDL, append=(knd, vnd, lens_out))
    torch.cuda.synchronize()
    assert e.item() == 0 and not err
    assert np.array_equal(lens_out.cpu().numpy(), lens_w)
    assert_attn_close(host16(out), want, dtype, "rope + GQA decode")
