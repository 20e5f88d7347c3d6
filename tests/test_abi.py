"""The C ABI library builds for sm_103a, loads, and exports every declared entry point.

CPU only: nothing here launches a kernel. Host-side argument checks that fail before
any CUDA call are exercised with fake (aligned, never dereferenced) pointers.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvdecode.h")


@pytest.fixture(scope="module")
def lib():
    from kv_cached_decode_gb300 import build, load_library

    build.build()
    return load_library()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(kvd_[a-z_0-9]+)\s*\(", text))


def test_header_declares_the_entry_points():
    want = {"kvd_kv_append", "kvd_decode_attn", "kvd_verify_attn", "kvd_greedy_accept",
            "kvd_beam_reorder_kv", "kvd_workspace_size", "kvd_status_string", "kvd_version",
            "kvd_prefill_attn", "kvd_rope", "kvd_beam_select", "kvd_kv_append_rope",
            "kvd_sample_accept"}
    assert want <= _declared()


def test_library_exports_every_declared_symbol(lib):
    for name in sorted(_declared()):
        assert hasattr(lib, name), name


def test_exports_are_plain_c_symbols(lib):
    out = os.popen(f"nm -D --defined-only {lib._name}").read()
    for name in _declared():
        assert re.search(rf"\bT {name}$", out, flags=re.M), name


def test_status_strings_and_version(lib):
    from kv_cached_decode_gb300 import STATUS_NAMES, kvd_status_string, kvd_version

    for code, name in STATUS_NAMES.items():
        assert kvd_status_string(code).startswith(name)
    assert kvd_status_string(99) == "unknown kvd_status"
    assert kvd_version() >= 100


def test_workspace_sizes_cover_the_counter_region(lib):
    from kv_cached_decode_gb300 import (KVD_OP_DECODE_ATTN, KVD_OP_GREEDY_ACCEPT,
                                        KVD_OP_VERIFY_ATTN, KVD_WS_COUNTER_BYTES,
                                        kvd_workspace_size)

    a = kvd_workspace_size(KVD_OP_DECODE_ATTN, 1, 20, 20, 1, 1, 1500)
    b = kvd_workspace_size(KVD_OP_VERIFY_ATTN, 1, 20, 20, 1, 5, 448)
    c = kvd_workspace_size(KVD_OP_GREEDY_ACCEPT, 1, qlen=5, vocab=51865)
    assert min(a, b, c) >= KVD_WS_COUNTER_BYTES
    # the 1500-frame cross attention merges its splits inside clusters: counters only
    assert a == KVD_WS_COUNTER_BYTES
    # one KV head over 32768 positions splits past a cluster and needs partials
    d = kvd_workspace_size(KVD_OP_DECODE_ATTN, 1, 1, 1, 1, 1, 32768)
    assert d >= KVD_WS_COUNTER_BYTES + 128 * 66 * 4
    # invalid arguments give 0
    assert kvd_workspace_size(KVD_OP_DECODE_ATTN, 1, 20, 3) == 0
    assert kvd_workspace_size(KVD_OP_VERIFY_ATTN, 1, 20, 20, 1, 17, 448) == 0
    assert kvd_workspace_size(KVD_OP_GREEDY_ACCEPT, 1, qlen=0, vocab=10) == 0


@pytest.mark.parametrize("shape", [
    # (batch, q heads, kv heads, rows per kv, qlen, length): few (row, KV head) units over
    # long ranges, the shapes whose launches may span several clusters per unit
    (1, 1, 1, 1, 1, 32768), (1, 2, 2, 1, 1, 32768), (1, 20, 4, 1, 1, 16384),
    (1, 20, 4, 1, 1, 32768), (2, 20, 4, 1, 1, 32768), (1, 8, 1, 1, 1, 16384),
    (1, 16, 1, 1, 1, 32768), (1, 16, 1, 1, 6, 65536), (5, 5, 5, 5, 1, 65536),
])
def test_workspace_size_covers_several_clusters_per_unit(lib, shape):
    """A launch over few long units may give each unit up to 8 clusters whose first CTAs
    merge through the workspace: the size the library reports must hold those 8 partials
    per (unit, query vector), 64 fp32 values and a (max, sum) pair each, after the
    counters."""
    from kv_cached_decode_gb300 import (KVD_OP_DECODE_ATTN, KVD_OP_VERIFY_ATTN,
                                        KVD_WS_COUNTER_BYTES, kvd_workspace_size)

    B, Hq, Hkv, rpk, qlen, L = shape
    op = KVD_OP_DECODE_ATTN if qlen == 1 else KVD_OP_VERIFY_ATTN
    got = kvd_workspace_size(op, B, Hq, Hkv, rpk, qlen, L)
    M = rpk * (Hq // Hkv) * qlen                  # query vectors per (row, KV head)
    mmax = 16 if M >= 2 else 1
    nsub = -(-M // mmax)
    msub = -(-M // nsub)
    units = (B // rpk) * Hkv * nsub
    slots = units * 8 * msub
    need = KVD_WS_COUNTER_BYTES + -(-(slots * 64 * 4) // 256) * 256 + slots * 2 * 4
    assert got >= need, (shape, got, need)


def _fake_cache(**kw):
    from kv_cached_decode_gb300 import Cache

    c = dict(k=0x10000, v=0x20000, stride_b=20 * 448 * 64, stride_h=448 * 64, stride_t=64,
             batch=1, n_kv_heads=20, head_dim=64, capacity=448)
    c.update(kw)
    return Cache(**c)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=128), 2),
    (dict(k=0), 1),
    (dict(k=0x10008), 1),         # not 16-byte aligned
    (dict(stride_t=60), 1),
    (dict(stride_h=448 * 64 + 4), 1),
    (dict(capacity=0), 1),
])
def test_host_rejects_bad_caches_before_touching_the_gpu(lib, kw, status):
    c = _fake_cache(**kw)
    q = ctypes.c_void_p(0x30000)
    r = lib.kvd_decode_attn(0, 1, 20, q, ctypes.byref(c), None, 10, None, 1, 0.125, q, None,
                            0, 0, None, None)
    assert r == status


def test_host_rejects_bad_shapes(lib):
    c = _fake_cache()
    q = ctypes.c_void_p(0x30000)
    # query heads not a multiple of KV heads
    assert lib.kvd_decode_attn(0, 1, 30, q, ctypes.byref(c), None, 10, None, 1, 0.125, q, None,
                               0, 0, None, None) == 1
    # batch not a multiple of rows_per_kv
    assert lib.kvd_decode_attn(0, 3, 20, q, ctypes.byref(c), None, 10, None, 2, 0.125, q, None,
                               0, 0, None, None) == 1
    # fixed length past the capacity
    assert lib.kvd_decode_attn(0, 1, 20, q, ctypes.byref(c), None, 449, None, 1, 0.125, q,
                               None, 0, 0, None, None) == 1
    # verify block longer than 16
    assert lib.kvd_verify_attn(0, 1, 20, 17, q, ctypes.byref(c), None, 10, None, 1, 1, 0.125,
                               q, None, 0, 0, None, None) == 2
    # append: lens_out aliasing lens_in
    lens = ctypes.c_void_p(0x40000)
    assert lib.kvd_kv_append(0, ctypes.byref(c), 1, 1, q, q, lens, lens, 0, None, None) == 1
    # beam larger than 8, rows not a multiple of beam
    arr = (type(c) * 1)(c)
    assert lib.kvd_beam_reorder_kv(0, arr, 1, 9, 9, lens, None, 4, 0, None, None) == 2
    assert lib.kvd_beam_reorder_kv(0, arr, 1, 7, 5, lens, None, 4, 0, None, None) == 1
    # accept: k out of range
    assert lib.kvd_greedy_accept(q, 1, 0, 100, q, q, q, None, None, q, 1 << 20, 0, None,
                                 None) == 2
    # fused append without lengths, or with lens_out aliasing lens
    from kv_cached_decode_gb300 import NewTokens

    app = NewTokens(0x50000, 0x60000, None)
    assert lib.kvd_decode_attn(0, 1, 20, q, ctypes.byref(c), None, 10, ctypes.byref(app), 1,
                               0.125, q, None, 0, 0, None, None) == 1
    app_alias = NewTokens(0x50000, 0x60000, 0x40000)
    assert lib.kvd_decode_attn(0, 1, 20, q, ctypes.byref(c), lens, 10, ctypes.byref(app_alias),
                               1, 0.125, q, None, 0, 0, None, None) == 1
    # a negative or NaN rotary base
    for base in (-1.0, float("nan"), float("inf")):
        app_rope = NewTokens(0x50000, 0x60000, None, base)
        assert lib.kvd_decode_attn(0, 1, 20, q, ctypes.byref(c), lens, 10,
                                   ctypes.byref(app_rope), 1, 0.125, q, None, 0, 0, None,
                                   None) == 1
    # empty batches are a no-op
    assert lib.kvd_decode_attn(0, 0, 20, None, ctypes.byref(c), None, 0, None, 1, 0.125, None,
                               None, 0, 0, None, None) == 0


def test_noalloc_rejects_bad_arguments_before_any_cuda_call(lib):
    # The no-workspace entry point runs every host check before it looks up its built-in
    # scratch or enqueues anything: on this GPU-less host, fake pointers with a bad
    # argument must come back as KVD_ERR_INVALID_ARG (a CUDA call would give
    # KVD_ERR_CUDA instead).
    c = _fake_cache()
    q = ctypes.c_void_p(0x30000)
    call = lib.kvd_decode_attn_noalloc
    assert call(0, 1, 30, q, ctypes.byref(c), None, 10, None, 1, 0.125, q, 0, None, None) == 1
    assert call(0, 1, 20, ctypes.c_void_p(0x30008), ctypes.byref(c), None, 10, None, 1, 0.125,
                q, 0, None, None) == 1                       # misaligned query
    assert call(0, 1, 20, q, ctypes.byref(c), None, 449, None, 1, 0.125, q, 0, None,
                None) == 1                                   # fixed length past capacity
    bad = _fake_cache(k=0)
    assert call(0, 1, 20, q, ctypes.byref(bad), None, 10, None, 1, 0.125, q, 0, None,
                None) == 1                                   # no K buffer
    assert call(0, 0, 20, None, ctypes.byref(c), None, 0, None, 1, 0.125, None, 0, None,
                None) == 0                                   # nothing to do


def test_prefill_host_rejects_bad_arguments(lib):
    c = _fake_cache()
    p = ctypes.c_void_p(0x30000)
    lens = ctypes.c_void_p(0x40000)
    # no prompt lengths
    assert lib.kvd_prefill_attn(0, 1, 20, 16, p, ctypes.byref(c), p, p, None, None, None,
                                0.125, 0.0, p, 0, None, None) == 1
    # query heads not a multiple of KV heads
    assert lib.kvd_prefill_attn(0, 1, 30, 16, p, ctypes.byref(c), p, p, None, lens, None,
                                0.125, 0.0, p, 0, None, None) == 1
    # lens_out aliasing lens_in, and a misaligned query pointer
    assert lib.kvd_prefill_attn(0, 1, 20, 16, p, ctypes.byref(c), p, p, lens, lens, lens,
                                0.125, 0.0, p, 0, None, None) == 1
    assert lib.kvd_prefill_attn(0, 1, 20, 16, ctypes.c_void_p(0x30008), ctypes.byref(c), p, p,
                                None, lens, None, 0.125, 0.0, p, 0, None, None) == 1
    # a bad cache, a bad dtype, and the empty cases
    bad = _fake_cache(head_dim=128)
    assert lib.kvd_prefill_attn(0, 1, 20, 16, p, ctypes.byref(bad), p, p, None, lens, None,
                                0.125, 0.0, p, 0, None, None) == 2
    assert lib.kvd_prefill_attn(7, 1, 20, 16, p, ctypes.byref(c), p, p, None, lens, None,
                                0.125, 0.0, p, 0, None, None) == 1
    assert lib.kvd_prefill_attn(0, 0, 20, 16, None, ctypes.byref(c), None, None, None, None,
                                None, 0.125, 0.0, None, 0, None, None) == 0
    assert lib.kvd_prefill_attn(0, 1, 20, 0, None, ctypes.byref(c), None, None, None, None,
                                None, 0.125, 0.0, None, 0, None, None) == 0
    # a negative rotary base
    assert lib.kvd_prefill_attn(0, 1, 20, 16, p, ctypes.byref(c), p, p, None, lens, None,
                                0.125, -1.0, p, 0, None, None) == 1


def test_rope_host_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(0x30000)
    assert lib.kvd_rope(0, 1, 4, p, 4, p, 2, None, 0.0, 0, None, None) == 1      # base 0
    assert lib.kvd_rope(0, 1, 4, ctypes.c_void_p(0x30002), 4, None, 0, None, 1e4, 0, None,
                        None) == 1                                               # misaligned
    assert lib.kvd_rope(0, 1, 4, p, 0, None, 0, None, 1e4, 0, None, None) == 1   # no heads
    assert lib.kvd_rope(5, 1, 4, p, 4, None, 0, None, 1e4, 0, None, None) == 1   # dtype
    assert lib.kvd_rope(0, 1, 4, None, 0, None, 0, None, 1e4, 0, None, None) == 0  # nothing


def test_beam_select_host_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(0x40000)

    def call(windows=1, beam=5, vocab=100, eot=99, n_sup=0, parent=p, row_token=None,
             logits=p):
        return lib.kvd_beam_select(logits, windows, beam, vocab, None, p, n_sup, None, 0, eot,
                                   0, row_token, None, parent, p, p, p, p, p, 0, None, None)

    assert call(beam=9) == 2                         # beam above 8
    assert call(beam=0) == 2
    assert call(vocab=5) == 1                        # vocab must exceed beam
    assert call(eot=100) == 1 and call(eot=-1) == 1  # EOT outside the vocabulary
    assert call(windows=-1) == 1
    assert call(windows=0) == 0                      # nothing to do
    assert call(windows=(1 << 24) + 1) == 2          # too many windows
    assert call(parent=None) == 1                    # no output at all
    assert call(vocab=524289, eot=0) == 2            # vocabulary too large
    assert call(logits=ctypes.c_void_p(0x40002)) == 1  # logits not 4-byte aligned
    assert lib.kvd_beam_select(p, 1, 5, 100, None, None, 3, None, 0, 99, 0, None, None, p, p,
                               p, p, p, p, 0, None, None) == 1  # suppression list missing
    assert lib.kvd_beam_select(p, 1, 5, 100, None, None, 0, None, 0, 99, 0, None, None, p,
                               None, p, p, p, p, 0, None, None) == 1  # partial walk outputs


def test_append_rope_host_rejects_bad_arguments(lib):
    c = _fake_cache()
    p = ctypes.c_void_p(0x30000)
    lens = ctypes.c_void_p(0x40000)
    for base in (0.0, -2.0, float("nan"), float("inf")):
        assert lib.kvd_kv_append_rope(0, ctypes.byref(c), 1, 1, p, p, lens, None, base, 0,
                                      None, None) == 1
    assert lib.kvd_kv_append_rope(0, ctypes.byref(c), 0, 1, None, None, None, None, 1e4, 0,
                                  None, None) == 0


def test_sample_accept_host_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(0x30000)

    def call(k=2, vocab=100, T=1.0, draft=p, batch=1, ws=ctypes.c_void_p(0x100000),
             ws_bytes=1 << 20):
        return lib.kvd_sample_accept(p, draft, p, batch, k, vocab, T, p, p, p, p, ws, ws_bytes,
                                     0, None, None)

    assert call(k=8) == 2                                  # more than 7 drafts
    assert call(k=-1) == 1
    for T in (0.0, -1.0, float("nan"), float("inf")):
        assert call(T=T) == 1                              # temperature must be > 0
    assert call(draft=None) == 1                           # drafts without a draft model
    assert call(k=0, draft=None, batch=0) == 0             # nothing to do
    assert call(vocab=0) == 1
    assert call(ws=None) == 3 and call(ws_bytes=1024) == 3  # workspace missing / too small
    from kv_cached_decode_gb300 import KVD_OP_SAMPLE_ACCEPT, KVD_WS_COUNTER_BYTES
    n = lib.kvd_workspace_size(KVD_OP_SAMPLE_ACCEPT, 16, 0, 0, 0, 5, 0, 51865)
    assert n >= KVD_WS_COUNTER_BYTES + 16 * 11 * 26 * 8  # (max, sum) per row and segment
    assert lib.kvd_workspace_size(KVD_OP_SAMPLE_ACCEPT, 16, 0, 0, 0, 8, 0, 51865) == 0


def test_binding_refuses_host_and_mistyped_tensors(lib):
    # The binding passes raw device addresses: a host tensor would reach a kernel as a
    # pointer into host memory, so it is refused before the library is called.
    import torch

    import kv_cached_decode_gb300 as kvd

    logits = torch.zeros(1, 3, 10, dtype=torch.float32)
    draft = torch.zeros(1, 2, dtype=torch.int32)
    n, nxt = torch.zeros(1, dtype=torch.int32), torch.zeros(1, dtype=torch.int32)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="logits must be a CUDA tensor"):
        kvd.kvd_greedy_accept(logits, draft, n, nxt, ws)
    with pytest.raises(ValueError, match="target must be a CUDA tensor"):
        kvd.kvd_sample_accept(logits[:, :1], torch.zeros(1), n, nxt, ws)
    with pytest.raises(ValueError, match="logits must be a CUDA tensor"):
        kvd.kvd_beam_select(torch.zeros(2, 10), 2)
