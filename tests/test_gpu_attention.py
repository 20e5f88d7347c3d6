"""GPU parity of decode attention (self, cross, split merge) and verify attention against the
fp64 oracle, through the C ABI. Tolerance: max-abs <= 1e-2, rel-Frobenius <= 5e-3."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import (assert_attn_close, dev16, dev_i32, host16, new_err, require_gpu)
from workloads import gen_cache, gen_lens_uniform, gen_new_kv, gen_queries, make_rng

pytestmark = pytest.mark.gpu

D = 64


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _kvd():
    import kv_cached_decode_gb300 as kvd

    return kvd


def run_attention(dtype, B, Hq, Hkv, cap, *, lens=None, fixed_len=0, rpk=1, qlen=1,
                  causal=False, verify=False, seed=0, q_std=0.125, kv_std=0.125, scale=0.125,
                  needles=(), repeat_check=True):
    """Run the GPU kernel and the oracle on the same seeded inputs; return both."""
    kvd = _kvd()
    rng = make_rng(seed)
    Bkv = B // rpk
    fill = lens if lens is not None else [fixed_len] * Bkv
    K, V = gen_cache(rng, Bkv, Hkv, cap, D, dtype, kv_std, lens=fill)
    q = gen_queries(rng, B, Hq, qlen, D, dtype, q_std)
    for (b, h, pos, gain) in needles:  # a key pointing along the query: a sharp peak
        qv = q[b * rpk, h * (Hq // Hkv), 0].view(np.float16 if dtype == "f16" else np.uint16)
        if dtype == "f16":
            K[b, h, pos] = (qv.astype(np.float64) * gain).astype(np.float16).view(np.uint16)
        else:
            K[b, h, pos] = qv  # bf16: reuse the query bits (score = |q|^2 * scale)
    want, err = oracle.attention(q, K, V, dtype, lens=lens, fixed_len=fixed_len,
                                 rows_per_kv=rpk, causal=causal, scale=scale)
    assert not err
    Kd, Vd, qd = dev16(K, dtype), dev16(V, dtype), dev16(q, dtype)
    out = torch.empty_like(qd)
    cache = kvd.make_cache(Kd, Vd)
    op = kvd.KVD_OP_VERIFY_ATTN if verify else kvd.KVD_OP_DECODE_ATTN
    bound = cap if lens is not None else fixed_len
    ws = kvd.new_workspace(kvd.kvd_workspace_size(op, B, Hq, Hkv, rpk, qlen, bound))
    lens_d = None if lens is None else dev_i32(lens)
    e = new_err()

    def call(o):
        if verify:
            kvd.kvd_verify_attn(qd, cache, o, ws, lens=lens_d, fixed_len=fixed_len,
                                rows_per_kv=rpk, causal=causal, scale=scale, dev_err=e)
        else:
            kvd.kvd_decode_attn(qd, cache, o, ws, lens=lens_d, fixed_len=fixed_len,
                                rows_per_kv=rpk, scale=scale, dev_err=e)

    call(out)
    torch.cuda.synchronize()
    assert e.item() == 0
    assert int(ws[: kvd.KVD_WS_COUNTER_BYTES].sum().item()) == 0, "counters not returned to 0"
    got = host16(out)
    if repeat_check:  # a fixed split order makes the result bit-reproducible
        out2 = torch.empty_like(qd)
        call(out2)
        torch.cuda.synchronize()
        assert np.array_equal(host16(out2), got)
    return got, want


# ------------------------------------------------------------------------- decode -------

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_tiny_layer_self_and_cross(dtype):
    got, want = run_attention(dtype, 1, 6, 6, 33, lens=np.array([33], np.int32), seed=1)
    assert_attn_close(got, want, dtype, "tiny self L=33")
    got, want = run_attention(dtype, 1, 6, 6, 1500, fixed_len=1500, seed=2)
    assert_attn_close(got, want, dtype, "tiny cross 1500")


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 128, 200, 447, 448])
def test_whisper_self_lengths(L):
    got, want = run_attention("f16", 1, 20, 20, 448, lens=np.array([L], np.int32), seed=L)
    assert_attn_close(got, want, "f16", f"self L={L}")


def test_whisper_cross_1500():
    got, want = run_attention("f16", 1, 20, 20, 1500, fixed_len=1500, seed=7)
    assert_attn_close(got, want, "f16", "cross")


def test_gqa_lm_ragged_bf16():
    rng = make_rng(4001)
    lens = gen_lens_uniform(rng, 16, 256, 2048) + 1
    got, want = run_attention("bf16", 16, 9, 3, 2112, lens=lens, seed=4002)
    assert_attn_close(got, want, "bf16", "gqa ragged")


def test_beam_rows_share_window_cross():
    got, want = run_attention("f16", 10, 20, 20, 1500, fixed_len=1500, rpk=5, seed=9)
    assert_attn_close(got, want, "f16", "beam cross")


@pytest.mark.parametrize("B,L", [(1, 128), (4, 2048), (16, 512), (1, 8192)])
def test_sweep_points_gqa_20_4(B, L):
    got, want = run_attention("f16", B, 20, 4, L + 1, lens=np.full(B, L, np.int32), seed=B + L)
    assert_attn_close(got, want, "f16", f"sweep B={B} L={L}")


def test_many_query_vectors_per_kv_head():
    # rows_per_kv 4 x group 3 = 12 query vectors per KV head: two query sub-blocks
    got, want = run_attention("bf16", 8, 6, 2, 300, lens=np.array([300, 17], np.int32), rpk=4,
                              seed=11)
    assert_attn_close(got, want, "bf16", "M=12")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_peaked_softmax(dtype):
    got, want = run_attention(dtype, 2, 8, 8, 700, lens=np.array([700, 333], np.int32),
                              q_std=3.0, seed=12)
    assert_attn_close(got, want, dtype, "peaked")


@pytest.mark.parametrize("pos", [0, 63, 64, 127, 999])
def test_needle_positions(pos):
    got, want = run_attention("f16", 1, 4, 4, 1000, fixed_len=1000, seed=13,
                              needles=[(0, 1, pos, 400.0)])
    assert_attn_close(got, want, "f16", f"needle {pos}")
    # the needle head's output is essentially that position's V
    assert np.max(np.abs(want[0, 1, 0])) > 0


def test_zero_length_rows_give_zeros():
    lens = np.array([0, 5, 0, 130], np.int32)
    got, want = run_attention("f16", 4, 4, 4, 130, lens=lens, seed=14)
    assert_attn_close(got, want, "f16", "zero rows")
    assert np.all(got[0] == 0) and np.all(got[2] == 0)


def test_length_past_capacity_sets_the_flag_and_skips():
    kvd = _kvd()
    rng = make_rng(15)
    K, V = gen_cache(rng, 2, 2, 64, D, "f16", 0.125)
    q = gen_queries(rng, 2, 2, 1, D, "f16", 0.125)
    Kd, Vd, qd = dev16(K, "f16"), dev16(V, "f16"), dev16(q, "f16")
    out = torch.full_like(qd, 7.0)
    e = new_err()
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_DECODE_ATTN, 2, 2, 2, 1, 1, 64))
    kvd.kvd_decode_attn(qd, kvd.make_cache(Kd, Vd), out, ws, lens=dev_i32([65, 64]), dev_err=e)
    torch.cuda.synchronize()
    assert e.item() == 16
    assert torch.all(out[0] == 7.0)  # the bad row is left as is
    want, _ = oracle.attention(q[1:], K[1:], V[1:], "f16", lens=np.array([64], np.int32))
    assert_attn_close(host16(out[1:]), want, "f16", "good row")


def test_strided_cache_view():
    """A cache that is a capacity slice of a larger allocation (padded strides)."""
    kvd = _kvd()
    rng = make_rng(16)
    Kbig, Vbig = gen_cache(rng, 2, 3, 96, D, "bf16", 0.125)
    K, V = Kbig[:, :, :80], Vbig[:, :, :80]
    lens = np.array([80, 41], np.int32)
    q = gen_queries(rng, 2, 3, 1, D, "bf16", 0.125)
    want, _ = oracle.attention(q, np.ascontiguousarray(K), np.ascontiguousarray(V), "bf16",
                               lens=lens)
    Kd = dev16(Kbig, "bf16")[:, :, :80]
    Vd = dev16(Vbig, "bf16")[:, :, :80]
    qd = dev16(q, "bf16")
    out = torch.empty_like(qd)
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_DECODE_ATTN, 2, 3, 3, 1, 1, 80))
    kvd.kvd_decode_attn(qd, kvd.make_cache(Kd, Vd), out, ws, lens=dev_i32(lens))
    torch.cuda.synchronize()
    assert_attn_close(host16(out), want, "bf16", "strided")


def test_workspace_too_small_is_rejected():
    """Two (row, head) units over 32768 positions merge through the workspace."""
    kvd = _kvd()
    K = torch.zeros(1, 2, 32768, D, dtype=torch.float16, device="cuda")
    q = torch.zeros(1, 2, 1, D, dtype=torch.float16, device="cuda")
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvd.KvdError) as ei:
        kvd.kvd_decode_attn(q, kvd.make_cache(K, K), q.clone(), ws, fixed_len=32768)
    assert ei.value.status == 3
    with pytest.raises(kvd.KvdError):
        kvd.kvd_decode_attn(q, kvd.make_cache(K, K), q.clone(), None, fixed_len=32768)


def test_beam_cross_eight_windows_register_variant():
    # 8 windows x beam 5 over 1500 frames: 160 (window, head) units, too many for
    # cluster splits at 2 blocks per SM; the 3-blocks-per-SM build halves each block's
    # tiles and runs instead
    got, want = run_attention("f16", 40, 20, 20, 1500, fixed_len=1500, rpk=5, seed=173)
    assert_attn_close(got, want, "f16", "beam cross, 8 windows")


# One query vector per KV head runs on the CUDA-core kernel when blocks stream several
# rounds of tiles (long caches); short caches go to the tensor-core kernel. These shapes
# keep the CUDA-core kernel's cluster merge, single-split store and fused append covered.
def test_decode_cuda_core_cluster_merge():
    # 80 (row, head) units over 2048 positions: clusters of 5 splits of 8 tiles
    lens = np.array([2048, 1900, 1, 1000], np.int32)
    got, want = run_attention("f16", 4, 20, 20, 2048, lens=lens, seed=170)
    assert_attn_close(got, want, "f16", "CUDA-core decode, cluster merge")


def test_decode_cuda_core_single_split():
    # 512 units fill the GPU by themselves: one block per unit, 8 tiles each
    rng = make_rng(171)
    lens = gen_lens_uniform(rng, 64, 1, 512)
    got, want = run_attention("bf16", 64, 8, 8, 512, lens=lens, seed=172)
    assert_attn_close(got, want, "bf16", "CUDA-core decode, one split")


# ------------------------------------------------------------------------- verify -------

@pytest.mark.parametrize("qlen", [5, 6])
@pytest.mark.parametrize("L", [0, 1, 59, 60, 443])
def test_verify_self_causal_whisper(qlen, L):
    if L + qlen > 448:
        pytest.skip("past n_text_ctx")
    got, want = run_attention("f16", 1, 20, 20, 448, lens=np.array([L + qlen], np.int32),
                              qlen=qlen, causal=True, verify=True, seed=100 + L + qlen)
    assert_attn_close(got, want, "f16", f"verify self L={L} q={qlen}")


def test_verify_cross_non_causal():
    got, want = run_attention("f16", 1, 20, 20, 1500, fixed_len=1500, qlen=5, causal=False,
                              verify=True, seed=120)
    assert_attn_close(got, want, "f16", "verify cross")


def test_verify_gqa_ragged_bf16():
    rng = make_rng(121)
    lens = gen_lens_uniform(rng, 16, 4, 2048)
    got, want = run_attention("bf16", 16, 9, 3, 2112, lens=lens, qlen=4, causal=True,
                              verify=True, seed=122)
    assert_attn_close(got, want, "bf16", "verify gqa")


def test_verify_large_block_splits_queries():
    # qlen 16 x group 3 = 48 query vectors per KV head: three tensor-core row blocks
    got, want = run_attention("f16", 2, 6, 2, 256, lens=np.array([256, 40], np.int32), qlen=16,
                              causal=True, verify=True, seed=123)
    assert_attn_close(got, want, "f16", "verify M=48")


def test_verify_block_longer_than_cache():
    got, want = run_attention("f16", 2, 4, 4, 64, lens=np.array([3, 0], np.int32), qlen=5,
                              causal=True, verify=True, seed=124)
    assert_attn_close(got, want, "f16", "len < qlen")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_verify_peaked(dtype):
    got, want = run_attention(dtype, 1, 8, 8, 448, lens=np.array([448], np.int32), qlen=5,
                              causal=True, verify=True, q_std=3.0, seed=125)
    assert_attn_close(got, want, dtype, "verify peaked")


def test_verify_single_token_equals_decode():
    a, want = run_attention("f16", 3, 8, 4, 300, lens=np.array([300, 1, 77], np.int32),
                            qlen=1, causal=True, verify=True, seed=126)
    b, _ = run_attention("f16", 3, 8, 4, 300, lens=np.array([300, 1, 77], np.int32), seed=126)
    assert_attn_close(a, want, "f16", "verify q=1")
    assert_attn_close(b, want, "f16", "decode")


# Few (row, head) units over a long range: one 16-block cluster per unit would leave each
# block 16 rounds of tiles, so the range is cut into 128 splits. With 2 units all 16
# clusters (8 per unit, 16 blocks each) are resident at once: each cluster merges on chip,
# and the last of a unit's 8 first CTAs to arrive merges their partials through the
# workspace.
def test_decode_workspace_merge_long_cache():
    got, want = run_attention("f16", 1, 2, 2, 32768, lens=np.array([32000], np.int32), seed=130)
    assert_attn_close(got, want, "f16", "decode 2 units x 8 clusters of 16 splits")


# 8 units over a long range: only about 2 clusters of 16 per unit can be resident at
# once, which would leave each block more tiles than plain splits do, so every block
# publishes its partial to the workspace and the last to arrive merges them (ragged rows:
# the second row's blocks past its length have no tiles).
def test_decode_workspace_merge_without_clusters():
    got, want = run_attention("f16", 2, 20, 4, 32768, lens=np.array([32768, 17001], np.int32),
                              seed=132)
    assert_attn_close(got, want, "f16", "decode 8 units, workspace merge of plain splits")


# Two rows over 32768 positions, the second only 3000 long: that row's clusters past the
# first hold no tiles at all, and their first CTAs publish empty partials (max -inf, sum
# 0) that the merge across clusters must weigh 0. bf16, one query vector per KV head (the
# CUDA-core build with the merge across clusters).
def test_decode_grouped_merge_empty_clusters():
    got, want = run_attention("bf16", 2, 1, 1, 32768, lens=np.array([32768, 3000], np.int32),
                              seed=133)
    assert_attn_close(got, want, "bf16", "decode, clusters past the length empty")


def test_verify_workspace_merge_sixteen_queries():
    # 16 query heads on one KV head, qlen 1: 16 query vectors per block, 128 splits
    got, want = run_attention("bf16", 1, 16, 1, 32768, lens=np.array([32768], np.int32), qlen=1,
                              causal=True, verify=True, seed=131)
    assert_attn_close(got, want, "bf16", "verify M=16 workspace merge")


# ----------------------------------------------------------------- fused append ---------

def run_fused(dtype, B, Hq, Hkv, cap, lens_in, qlen, *, verify, seed, flags=0):
    """Attention with the new tokens appended in the same launch, against the oracle's
    kv_append followed by attention over the appended cache."""
    kvd = _kvd()
    rng = make_rng(seed)
    lens_in = np.asarray(lens_in, np.int32)
    K, V = gen_cache(rng, B, Hkv, cap, D, dtype, 0.125, lens=lens_in)
    kn, vn = gen_new_kv(rng, B, Hkv, qlen, D, dtype, 0.125)
    q = gen_queries(rng, B, Hq, qlen, D, dtype, 0.125)
    Kd, Vd = dev16(K, dtype), dev16(V, dtype)
    Kw, Vw = K.copy(), V.copy()
    lens_out_w, err = oracle.kv_append(Kw, Vw, kn, vn, lens_in, dtype)
    want, _ = oracle.attention(q, Kw, Vw, dtype, lens=lens_out_w, causal=verify)
    qd = dev16(q, dtype)
    out = torch.empty_like(qd)
    lens_out = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    op = kvd.KVD_OP_VERIFY_ATTN if verify else kvd.KVD_OP_DECODE_ATTN
    ws = kvd.new_workspace(kvd.kvd_workspace_size(op, B, Hq, Hkv, 1, qlen, cap))
    e = new_err()
    app = (dev16(kn, dtype), dev16(vn, dtype), lens_out)
    if verify:
        kvd.kvd_verify_attn(qd, kvd.make_cache(Kd, Vd), out, ws, lens=dev_i32(lens_in),
                            causal=True, flags=flags, dev_err=e, append=app)
    else:
        kvd.kvd_decode_attn(qd, kvd.make_cache(Kd, Vd), out, ws, lens=dev_i32(lens_in),
                            flags=flags, dev_err=e, append=app)
    torch.cuda.synchronize()
    return host16(out), want, host16(Kd), host16(Vd), Kw, Vw, lens_out.cpu().numpy(), \
        lens_out_w, e.item(), err


# The new token appended inside a launch whose units span several clusters (2 units over
# 32768 positions): the block whose slab holds position 30000 writes it to the cache and
# attends to it, and its cluster's partial reaches the merge across clusters.
@pytest.mark.parametrize("flags", [0, 3])  # plain, and PDL + early K/V
def test_decode_fused_append_several_clusters_per_unit(flags):
    got, want, Kg, Vg, Kw, Vw, lo, low, e, err = run_fused(
        "f16", 1, 2, 2, 32768, [30000], 1, verify=False, seed=134, flags=flags)
    assert e == 0 and not err
    assert np.array_equal(Kg, Kw) and np.array_equal(Vg, Vw)
    assert np.array_equal(lo, low)
    assert_attn_close(got, want, "f16", "fused decode, several clusters per unit")


@pytest.mark.parametrize("flags", [0, 3])  # plain, and PDL + early K/V
def test_decode_fused_append_whisper_self(flags):
    got, want, Kg, Vg, Kw, Vw, lo, low, e, err = run_fused(
        "f16", 1, 20, 20, 448, [447], 1, verify=False, seed=140, flags=flags)
    assert e == 0 and not err
    assert np.array_equal(Kg, Kw) and np.array_equal(Vg, Vw)
    assert np.array_equal(lo, low)
    assert_attn_close(got, want, "f16", "fused decode")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_decode_fused_append_ragged_tile_edges(dtype):
    lens = [0, 63, 64, 127, 128, 300, 511, 1]
    got, want, Kg, Vg, Kw, Vw, lo, low, e, err = run_fused(
        dtype, 8, 4, 4, 512, lens, 1, verify=False, seed=141)
    assert e == 0 and not err
    assert np.array_equal(Kg, Kw) and np.array_equal(Vg, Vw) and np.array_equal(lo, low)
    assert_attn_close(got, want, dtype, "fused decode ragged")


def test_decode_fused_append_gqa_tensor_cores():
    rng = make_rng(142)
    lens = gen_lens_uniform(rng, 16, 256, 2048)
    got, want, Kg, Vg, Kw, Vw, lo, low, e, err = run_fused(
        "bf16", 16, 9, 3, 2112, lens, 1, verify=False, seed=143, flags=3)
    assert e == 0 and np.array_equal(Kg, Kw) and np.array_equal(lo, low)
    assert_attn_close(got, want, "bf16", "fused gqa")


@pytest.mark.parametrize("L", [0, 59, 60, 62, 443])
@pytest.mark.parametrize("flags", [0, 3])
def test_verify_fused_append_block(L, flags):
    # L = 62: the five new rows straddle the boundary between two 64-position tiles
    got, want, Kg, Vg, Kw, Vw, lo, low, e, err = run_fused(
        "f16", 1, 20, 20, 448, [L], 5, verify=True, seed=150 + L, flags=flags)
    assert e == 0 and not err
    assert np.array_equal(Kg, Kw) and np.array_equal(Vg, Vw) and np.array_equal(lo, low)
    assert_attn_close(got, want, "f16", f"fused verify L={L}")


@pytest.mark.parametrize("flags", [0, 3])
def test_decode_fused_append_cuda_core_path(flags):
    got, want, Kg, Vg, Kw, Vw, lo, low, e, err = run_fused(
        "bf16", 4, 20, 20, 2048, [2047, 1000, 63, 0], 1, verify=False, seed=144, flags=flags)
    assert e == 0 and not err
    assert np.array_equal(Kg, Kw) and np.array_equal(Vg, Vw) and np.array_equal(lo, low)
    assert_attn_close(got, want, "bf16", "fused decode, CUDA cores")


def test_fused_append_overflow_leaves_row_untouched():
    got, want, Kg, Vg, Kw, Vw, lo, low, e, err = run_fused(
        "f16", 2, 2, 2, 64, [62, 10], 3, verify=True, seed=160)
    assert e == 16 and err == {16}
    assert np.array_equal(Kg, Kw) and np.array_equal(lo, low)  # row 0 untouched, len kept


def test_pdl_chain_on_one_stream():
    """append -> self decode -> cross decode -> fused verify, all with PDL (cross and
    verify with early K/V): every kernel must see its predecessor's writes."""
    kvd = _kvd()
    rng = make_rng(170)
    H, cap, F = 8, 256, 1500
    lens = np.array([200, 77], np.int32)
    K, V = gen_cache(rng, 2, H, cap, D, "f16", 0.125, lens=lens)
    Kx, Vx = gen_cache(rng, 2, H, F, D, "f16", 0.125)
    kn, vn = gen_new_kv(rng, 2, H, 1, D, "f16", 0.125)
    kb, vb = gen_new_kv(rng, 2, H, 5, D, "f16", 0.125)
    q1 = gen_queries(rng, 2, H, 1, D, "f16", 0.125)
    q5 = gen_queries(rng, 2, H, 5, D, "f16", 0.125)
    # oracle: append 1, decode self, decode cross, append 5, causal verify
    Kw, Vw = K.copy(), V.copy()
    l1, _ = oracle.kv_append(Kw, Vw, kn, vn, lens, "f16")
    w_self, _ = oracle.attention(q1, Kw, Vw, "f16", lens=l1)
    w_cross, _ = oracle.attention(q1, Kx, Vx, "f16", fixed_len=F)
    l2, _ = oracle.kv_append(Kw, Vw, kb, vb, l1, "f16")
    w_ver, _ = oracle.attention(q5, Kw, Vw, "f16", lens=l2, causal=True)
    # GPU
    Kd, Vd = dev16(K, "f16"), dev16(V, "f16")
    cache, xcache = kvd.make_cache(Kd, Vd), kvd.make_cache(dev16(Kx, "f16"), dev16(Vx, "f16"))
    l1d = torch.zeros(2, dtype=torch.int32, device="cuda")
    l2d = torch.zeros(2, dtype=torch.int32, device="cuda")
    q1d, q5d = dev16(q1, "f16"), dev16(q5, "f16")
    o_self, o_cross = torch.empty_like(q1d), torch.empty_like(q1d)
    o_ver = torch.empty_like(q5d)
    ws = kvd.new_workspace(kvd.kvd_workspace_size(kvd.KVD_OP_VERIFY_ATTN, 2, H, H, 1, 5, F))
    e = new_err()
    P, EK = kvd.KVD_FLAG_PDL, kvd.KVD_FLAG_PDL | kvd.KVD_FLAG_EARLY_KV
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        kvd.kvd_kv_append(cache, dev16(kn, "f16"), dev16(vn, "f16"), dev_i32(lens), l1d,
                          flags=P, dev_err=e)
        kvd.kvd_decode_attn(q1d, cache, o_self, ws, lens=l1d, flags=P, dev_err=e)
        kvd.kvd_decode_attn(q1d, xcache, o_cross, ws, fixed_len=F, flags=EK, dev_err=e)
        kvd.kvd_verify_attn(q5d, cache, o_ver, ws, lens=l1d, causal=True, flags=P, dev_err=e,
                            append=(dev16(kb, "f16"), dev16(vb, "f16"), l2d))
    torch.cuda.synchronize()
    assert e.item() == 0
    assert np.array_equal(l2d.cpu().numpy(), l2)
    assert np.array_equal(host16(Kd), Kw) and np.array_equal(host16(Vd), Vw)
    assert_attn_close(host16(o_self), w_self, "f16", "chain self")
    assert_attn_close(host16(o_cross), w_cross, "f16", "chain cross")
    assert_attn_close(host16(o_ver), w_ver, "f16", "chain verify")
