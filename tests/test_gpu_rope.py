"""Rotary encoding on the GPU (kvd_rope, and inside the attention call) against the
fp64 oracle.

Each rotated value must lie within one unit in the last place of the storage type of
the oracle's value, plus the fp32 angle's error times the pair's norm: the angle
pos * theta (theta <= 1) is formed from exp2f (<= 2 ulp) and one rounded product, so
its absolute error is below 2.5e-7 * pos; sin/cos add about 1e-6. End
to end, a decode or verify step whose queries and new keys are rotated at their
absolute positions must match the oracle's rotation (rounded to the storage type)
followed by its append and attention, within the attention tolerance. The rotation
inside the attention call must give the same bits as kvd_rope followed by the call:
outputs, caches and lengths.
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


def _angle_tol(pos):
    """Bound of the fp32 rotation's error per unit of pair norm at position pos."""
    return 2.5e-7 * (np.asarray(pos, np.float64) + 1) + 1e-6


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
        pos = (pos0[:, None, None, None] + np.arange(x.shape[2])[None, None, :, None])
        assert np.all(np.abs(got - want) <= _ulp(want, dtype) + _angle_tol(pos) * pair)
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


def _fused_vs_separate(dtype, B, Hq, Hkv, cap, lens, qlen, seed, *, verify=False):
    """The rotation inside the attention call against kvd_rope + the same call: the
    outputs, the caches and the lengths must be bit-identical."""
    import kv_cached_decode_gb300 as kvd

    rng = make_rng(seed)
    lens = np.asarray(lens, np.int32)
    K, V = gen_cache(rng, B, Hkv, cap, D, dtype, 0.125, lens=lens)
    kn, vn = gen_new_kv(rng, B, Hkv, qlen, D, dtype, 0.125)
    q = gen_queries(rng, B, Hq, qlen, D, dtype, 0.125)
    results = []
    for fused in (False, True):
        qd, knd, vnd = dev16(q, dtype), dev16(kn, dtype), dev16(vn, dtype)
        Kd, Vd = dev16(K, dtype), dev16(V, dtype)
        lens_d = dev_i32(lens)
        lens_out = torch.zeros_like(lens_d)
        out = torch.full_like(qd, 7.0)
        op = kvd.KVD_OP_VERIFY_ATTN if verify else kvd.KVD_OP_DECODE_ATTN
        ws = kvd.new_workspace(kvd.kvd_workspace_size(op, B, Hq, Hkv, 1, qlen, cap))
        e = new_err()
        if not fused:
            kvd.kvd_rope(qd, knd, lens_d)
        app = (knd, vnd, lens_out, 10000.0) if fused else (knd, vnd, lens_out)
        if verify:
            kvd.kvd_verify_attn(qd, kvd.make_cache(Kd, Vd), out, ws, lens=lens_d, causal=True,
                                dev_err=e, append=app)
        else:
            kvd.kvd_decode_attn(qd, kvd.make_cache(Kd, Vd), out, ws, lens=lens_d, dev_err=e,
                                append=app)
        torch.cuda.synchronize()
        assert e.item() == 0
        results.append((host16(out), host16(Kd), host16(Vd), lens_out.cpu().numpy()))
    for a, b in zip(*results):
        assert np.array_equal(a, b)
    # and against the oracle: rotate (rounded to the storage type), append, attend
    q_r = _round_bits(oracle.rope(q, dtype, lens), dtype)
    kn_r = _round_bits(oracle.rope(kn, dtype, lens), dtype)
    Kw, Vw = K.copy(), V.copy()
    lens_w, err = oracle.kv_append(Kw, Vw, kn_r, vn, lens, dtype)
    want, _ = oracle.attention(q_r, Kw, Vw, dtype, lens=lens_w, causal=verify)
    assert not err
    # the cache: unchanged outside the appended rows; there, the rotated keys within the
    # tolerance of the stand-alone rotation (fp32 on the GPU, fp64 in the oracle)
    Kg = results[1][1]
    new_rows = np.zeros(Kg.shape, bool)
    for b in range(B):
        new_rows[b, :, lens[b]:lens[b] + qlen] = True
    assert np.array_equal(Kg[~new_rows], Kw[~new_rows])
    want_k = oracle.rope(kn, dtype, lens)
    got_k = np.stack([_to_f64(Kg[b, :, lens[b]:lens[b] + qlen], dtype) for b in range(B)])
    xf = _to_f64(kn, dtype)
    pair = np.sqrt(xf[..., :32] ** 2 + xf[..., 32:] ** 2)
    pair = np.concatenate([pair, pair], axis=-1)
    pos = lens[:, None, None, None] + np.arange(qlen)[None, None, :, None]
    assert np.all(np.abs(got_k - want_k) <= _ulp(want_k, dtype) + _angle_tol(pos) * pair)
    assert_attn_close(results[1][0], want, dtype, "fused rotary encoding")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_fused_rope_gqa_decode(dtype):
    # grouped heads: the tensor-core kernel
    _fused_vs_separate(dtype, 4, 9, 3, 1100, [300, 1, 1000, 64], 1, seed=910)


def test_fused_rope_mha_decode_short_and_long():
    # one query per KV head: a short cache (one round of tiles) and a long one (the
    # CUDA-core kernel streams several rounds)
    _fused_vs_separate("f16", 2, 8, 8, 4200, [100, 40], 1, seed=911)
    _fused_vs_separate("f16", 2, 8, 8, 4200, [4100, 3000], 1, seed=912)


def test_fused_rope_causal_verify_block():
    # five tokens at positions lens + 0..4, causal, GQA
    _fused_vs_separate("bf16", 3, 6, 2, 700, [0, 250, 600], 5, seed=913, verify=True)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_append_rope_equals_rope_then_append(dtype):
    import kv_cached_decode_gb300 as kvd

    rng = make_rng(920)
    B, H, cap, q = 3, 4, 300, 5
    lens = np.array([0, 17, 290], np.int32)
    K, V = gen_cache(rng, B, H, cap, D, dtype, 0.125, lens=lens)
    kn, vn = gen_new_kv(rng, B, H, q, D, dtype, 0.125)
    caches = []
    for fused in (False, True):
        Kd, Vd = dev16(K, dtype), dev16(V, dtype)
        knd, vnd = dev16(kn, dtype), dev16(vn, dtype)
        lens_d, lens_out = dev_i32(lens), torch.zeros(B, dtype=torch.int32, device="cuda")
        e = new_err()
        if fused:
            kvd.kvd_kv_append_rope(kvd.make_cache(Kd, Vd), knd, vnd, lens_d, lens_out,
                                   rope_base=10000.0, dev_err=e)
        else:
            kvd.kvd_rope(None, knd, lens_d)
            kvd.kvd_kv_append(kvd.make_cache(Kd, Vd), knd, vnd, lens_d, lens_out, dev_err=e)
        torch.cuda.synchronize()
        assert e.item() == 0
        caches.append((host16(Kd), host16(Vd), lens_out.cpu().numpy()))
    for a, b in zip(*caches):
        assert np.array_equal(a, b)
    assert np.array_equal(caches[1][2], lens + q)
    # the appended keys against the oracle's rotation
    want_k = oracle.rope(kn, dtype, lens)
    got_k = np.stack([_to_f64(caches[1][0][b, :, lens[b]:lens[b] + q], dtype) for b in range(B)])
    xf = _to_f64(kn, dtype)
    pair = np.sqrt(xf[..., :32] ** 2 + xf[..., 32:] ** 2)
    pair = np.concatenate([pair, pair], axis=-1)
    pos = lens[:, None, None, None] + np.arange(q)[None, None, :, None]
    assert np.all(np.abs(got_k - want_k) <= _ulp(want_k, dtype) + _angle_tol(pos) * pair)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_rope_equals_rope_then_prefill(dtype):
    import kv_cached_decode_gb300 as kvd

    rng = make_rng(921)
    B, Hq, Hkv, cap, T = 3, 6, 2, 400, 150
    lens_in = np.array([0, 40, 200], np.int32)
    plens = np.array([150, 1, 97], np.int32)
    K, V = gen_cache(rng, B, Hkv, cap, D, dtype, 0.125, lens=lens_in)
    kn, vn = gen_new_kv(rng, B, Hkv, T, D, dtype, 0.125)
    q = gen_queries(rng, B, Hq, T, D, dtype, 0.125)
    res = []
    for fused in (False, True):
        Kd, Vd = dev16(K, dtype), dev16(V, dtype)
        qd, knd, vnd = dev16(q, dtype), dev16(kn, dtype), dev16(vn, dtype)
        li, pl = dev_i32(lens_in), dev_i32(plens)
        lens_out = torch.zeros(B, dtype=torch.int32, device="cuda")
        out = torch.full_like(qd, 3.0)
        e = new_err()
        if not fused:
            kvd.kvd_rope(qd, knd, li)
        kvd.kvd_prefill_attn(qd, kvd.make_cache(Kd, Vd), knd, vnd, pl, out, lens_in=li,
                             lens_out=lens_out, rope_base=10000.0 if fused else 0.0, dev_err=e)
        torch.cuda.synchronize()
        assert e.item() == 0
        res.append((host16(out), host16(Kd), host16(Vd), lens_out.cpu().numpy()))
    for a, b in zip(*res):
        assert np.array_equal(a, b)
    # against the oracle: rotate (rounded), append, causal attention per row
    q_r = _round_bits(oracle.rope(q, dtype, lens_in), dtype)
    kn_r = _round_bits(oracle.rope(kn, dtype, lens_in), dtype)
    Kw, Vw = K.copy(), V.copy()
    want = np.zeros((B, Hq, T, D))
    for b in range(B):
        n = plens[b]
        Kw[b, :, lens_in[b]:lens_in[b] + n] = kn_r[b, :, :n]
        Vw[b, :, lens_in[b]:lens_in[b] + n] = vn[b, :, :n]
        w, err = oracle.attention(q_r[b:b + 1, :, :n], Kw[b:b + 1], Vw[b:b + 1], dtype,
                                  lens=np.array([lens_in[b] + n], np.int32), causal=True)
        assert not err
        want[b, :, :n] = w[0]
    assert_attn_close(res[1][0], want, dtype, "prefill with rotary encoding")


def test_fused_rope_without_workspace():
    # the no-workspace entry point takes the same rotation: same bits as with a workspace
    import kv_cached_decode_gb300 as kvd

    rng = make_rng(930)
    B, Hq, Hkv, cap = 4, 9, 3, 700
    lens = np.array([5, 640, 300, 64], np.int32)
    K, V = gen_cache(rng, B, Hkv, cap, D, "bf16", 0.125, lens=lens)
    kn, vn = gen_new_kv(rng, B, Hkv, 1, D, "bf16", 0.125)
    q = gen_queries(rng, B, Hq, 1, D, "bf16", 0.125)
    res = []
    for noalloc in (False, True):
        Kd, Vd = dev16(K, "bf16"), dev16(V, "bf16")
        qd, knd, vnd = dev16(q, "bf16"), dev16(kn, "bf16"), dev16(vn, "bf16")
        lens_d, lens_out = dev_i32(lens), torch.zeros(B, dtype=torch.int32, device="cuda")
        out = torch.empty_like(qd)
        e = new_err()
        app = (knd, vnd, lens_out, 500000.0)
        if noalloc:
            kvd.kvd_decode_attn_noalloc(qd, kvd.make_cache(Kd, Vd), out, lens=lens_d, dev_err=e,
                                        append=app)
        else:
            ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_DECODE_ATTN, B, Hq, Hkv, 1,
                                                          1, cap))
            kvd.kvd_decode_attn(qd, kvd.make_cache(Kd, Vd), out, ws, lens=lens_d, dev_err=e,
                                append=app)
        torch.cuda.synchronize()
        assert e.item() == 0
        res.append((host16(out), host16(Kd), lens_out.cpu().numpy()))
    for a, b in zip(*res):
        assert np.array_equal(a, b)
