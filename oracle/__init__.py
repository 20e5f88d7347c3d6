"""fp64 CPU oracle for the KV-cached decoder step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library never imports, links or
runs it, and it imports nothing from the product library.

``kvd_oracle.c`` holds the definitions (append, attention, greedy accept, beam
reorder, rotary encoding, logit filters with the beam-search step, temperature sampling
with stochastic speculative acceptance); this module marshals numpy arrays into it. ``tiny_model.py`` builds a
small fp64 transformer on top of these functions for the end-to-end invariants
(cached == recomputed, speculative == greedy, beam reorder == per-beam recompute).

Every oracle function here is pinned by a ``-m "not gpu"`` test against something
other than itself: exhaustive number-format decoding against numpy, closed forms,
brute force, ``torch`` CPU attention and independent numpy recomputation, the
worked example of the speculative-decoding pages, and the tiny-model invariants.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERR_CODES = {1: 16, 2: 17, 4: 18, 8: 19}  # oracle bit -> status code
DTYPE_CODE = {"f16": 0, "bf16": 1, "f64": 2}


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc (plain -O2, no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # KVD_ORACLE_LIB lets the mutation test point the wrappers at a copy of the
            # oracle built with a deliberately planted mistake.
            path = os.environ.get("KVD_ORACLE_LIB") or build()
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_int64
            lib.kvo_decode_f16.argtypes = [ctypes.c_uint16]
            lib.kvo_decode_f16.restype = ctypes.c_double
            lib.kvo_decode_bf16.argtypes = [ctypes.c_uint16]
            lib.kvo_decode_bf16.restype = ctypes.c_double
            lib.kvo_kv_append.argtypes = [I, I, I, I, I, I, P, P, L, L, L, P, P, P, P]
            lib.kvo_kv_append.restype = ctypes.c_uint
            lib.kvo_attention.argtypes = [I, I, I, I, I, P, I, I, P, P, L, L, L, P, I, I, I,
                                          ctypes.c_double, P]
            lib.kvo_attention.restype = ctypes.c_uint
            lib.kvo_greedy_accept.argtypes = [I, I, I, P, P, P, P, P, P]
            lib.kvo_greedy_accept.restype = ctypes.c_uint
            lib.kvo_beam_reorder.argtypes = [I, I, I, I, I, I, I, P, P, P, L, L, L]
            lib.kvo_beam_reorder.restype = ctypes.c_uint
            lib.kvo_rope.argtypes = [I, I, I, I, I, P, P, ctypes.c_double, P]
            lib.kvo_rope.restype = None
            lib.kvo_beam_select.argtypes = [I, I, I, P, P, P, I, P, I, I, I, P, P, P, P, P, P,
                                            P, P]
            lib.kvo_beam_select.restype = ctypes.c_uint
            lib.kvo_sample_accept.argtypes = [I, I, I, P, P, P, ctypes.c_double, P, P, P, P]
            lib.kvo_sample_accept.restype = ctypes.c_uint
            _lib = lib
    return _lib


def _errs(mask: int) -> set:
    return {code for bit, code in ERR_CODES.items() if mask & bit}


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check_storage(a: np.ndarray, dtype: str):
    want = np.float64 if dtype == "f64" else np.uint16
    if a.dtype != want:
        raise TypeError(f"{dtype} data must be stored as {np.dtype(want).name}, got {a.dtype}")


def _elem_strides(a: np.ndarray):
    """Element strides of a 4-D cache array; the innermost stride must be 1."""
    st = tuple(s // a.itemsize for s in a.strides)
    if st[3] != 1:
        raise ValueError("head_dim must be the contiguous axis")
    return st[0], st[1], st[2]


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Decode uint16 fp16/bf16 bit patterns to float64 with the oracle's decoder."""
    lib = _load()
    fn = lib.kvo_decode_f16 if dtype == "f16" else lib.kvo_decode_bf16
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    out = np.fromiter((fn(int(x)) for x in flat), dtype=np.float64, count=flat.size)
    return out.reshape(np.shape(bits))


def kv_append(k_cache, v_cache, k_new, v_new, lens_in, dtype: str):
    """Append ``k_new/v_new [B,H,q,D]`` at positions ``lens_in[b]..`` (in place).

    Returns ``(lens_out, errors)``.
    """
    lib = _load()
    _check_storage(k_cache, dtype)
    B, H, cap, D = k_cache.shape
    q = k_new.shape[2]
    k_new = np.ascontiguousarray(k_new)
    v_new = np.ascontiguousarray(v_new)
    lens_in = np.ascontiguousarray(lens_in, dtype=np.int32)
    lens_out = np.empty_like(lens_in)
    sb, sh, st = _elem_strides(k_cache)
    assert _elem_strides(v_cache) == (sb, sh, st)
    m = lib.kvo_kv_append(DTYPE_CODE[dtype], B, H, cap, D, q, _ptr(k_cache), _ptr(v_cache),
                          sb, sh, st, _ptr(k_new), _ptr(v_new), _ptr(lens_in), _ptr(lens_out))
    return lens_out, _errs(m)


def attention(q, k_cache, v_cache, dtype: str, *, lens=None, fixed_len: int = 0,
              rows_per_kv: int = 1, causal: bool = False, scale: float = 0.125):
    """Attention of ``q [B,Hq,nq,D]`` over the cache ``[Bkv,Hkv,cap,D]``.

    Returns ``(out float64 [B,Hq,nq,D], errors)``.
    """
    lib = _load()
    _check_storage(k_cache, dtype)
    B, Hq, nq, D = q.shape
    _, Hkv, cap, D2 = k_cache.shape
    assert D == D2 and Hq % Hkv == 0
    q = np.ascontiguousarray(q)
    sb, sh, st = _elem_strides(k_cache)
    assert _elem_strides(v_cache) == (sb, sh, st)
    lens_arr = None if lens is None else np.ascontiguousarray(lens, dtype=np.int32)
    out = np.zeros((B, Hq, nq, D), dtype=np.float64)
    m = lib.kvo_attention(DTYPE_CODE[dtype], B, Hq, nq, D, _ptr(q), Hkv, cap,
                          _ptr(k_cache), _ptr(v_cache), sb, sh, st, _ptr(lens_arr),
                          int(fixed_len), int(rows_per_kv), int(bool(causal)),
                          float(scale), _ptr(out))
    return out, _errs(m)


def greedy_accept(logits, draft):
    """Greedy accept on fp32 ``logits [B,k+1,V]`` and int32 ``draft [B,k]``.

    Returns ``(n_accepted [B], next_token [B], n_min, argmax [B,k+1], errors)``.
    """
    lib = _load()
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    draft = np.ascontiguousarray(draft, dtype=np.int32)
    B, k1, V = logits.shape
    k = k1 - 1
    assert draft.shape == (B, k)
    n = np.empty(B, np.int32)
    nxt = np.empty(B, np.int32)
    nmin = np.empty(1, np.int32)
    amax = np.empty((B, k1), np.int32)
    m = lib.kvo_greedy_accept(B, k, V, _ptr(logits), _ptr(draft), _ptr(n), _ptr(nxt),
                              _ptr(nmin), _ptr(amax))
    return n, nxt, int(nmin[0]), amax, _errs(m)


def beam_reorder(cache, parent, beam: int, length: int, dtype: str):
    """Out-of-place reorder of one layer's K or V ``[R,H,cap,D]`` by ``parent``.

    Returns ``(new_cache, errors)``.
    """
    lib = _load()
    _check_storage(cache, dtype)
    cache = np.ascontiguousarray(cache)
    R, H, cap, D = cache.shape
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    dst = np.empty_like(cache)
    sb, sh, st = _elem_strides(cache)
    m = lib.kvo_beam_reorder(DTYPE_CODE[dtype], R, beam, H, cap, D, int(length),
                             _ptr(parent), _ptr(cache), _ptr(dst), sb, sh, st)
    return dst, _errs(m)


def rope(x, dtype: str, pos0=None, base: float = 10000.0):
    """Rotary encoding of ``x [B,H,n,D]`` (fp16/bf16 bits, or float64 with dtype "f64"),
    token j of row b at position ``pos0[b] + j``. Returns float64, same shape."""
    lib = _load()
    _check_storage(x, dtype)
    B, H, n, D = x.shape
    x = np.ascontiguousarray(x)
    p0 = None if pos0 is None else np.ascontiguousarray(pos0, dtype=np.int32)
    y = np.empty(x.shape, dtype=np.float64)
    code = {"f16": 0, "bf16": 1, "f64": 2}[dtype]
    lib.kvo_rope(code, B, H, n, D, _ptr(x), _ptr(p0), float(base), _ptr(y))
    return y


def beam_select(logits, beam: int, *, cum=None, suppress=(), blank=(), eot: int = 0,
                first_step: bool = False, walk: bool = True):
    """Logit filters and one beam-search step on fp32 ``logits [rows, vocab]``.

    Returns a dict: ``row_token``/``row_logprob [rows, beam+1]`` (each row's beam+1 best
    tokens after the filters), and with ``walk``: ``parent``/``token``/``new_cum
    [rows]`` (kept continuations, per window best first), ``n_fin [windows]``,
    ``fin_parent``/``fin_score [rows]``; plus ``errors``.
    """
    lib = _load()
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    rows, V = logits.shape
    assert rows % beam == 0
    kk = beam + 1
    cum_a = None if cum is None else np.ascontiguousarray(cum, dtype=np.float32)
    sup = np.ascontiguousarray(suppress, dtype=np.int32)
    blk = np.ascontiguousarray(blank, dtype=np.int32)
    r = {"row_token": np.empty((rows, kk), np.int32),
         "row_logprob": np.empty((rows, kk), np.float64)}
    if walk:
        r.update(parent=np.empty(rows, np.int32), token=np.empty(rows, np.int32),
                 new_cum=np.empty(rows, np.float64), n_fin=np.empty(rows // beam, np.int32),
                 fin_parent=np.empty(rows, np.int32), fin_score=np.empty(rows, np.float64))
    g = r.get
    m = lib.kvo_beam_select(rows, beam, V, _ptr(logits), _ptr(cum_a), _ptr(sup), sup.size,
                            _ptr(blk), blk.size, int(eot), int(bool(first_step)),
                            _ptr(r["row_token"]), _ptr(r["row_logprob"]), _ptr(g("parent")),
                            _ptr(g("token")), _ptr(g("new_cum")), _ptr(g("n_fin")),
                            _ptr(g("fin_parent")), _ptr(g("fin_score")))
    r["errors"] = _errs(m)
    return r


def sample_accept(target, temperature: float, u, *, draft=None, drafts=None, r=None):
    """Temperature sampling (k = 0) or stochastic speculative acceptance of k drafts.

    target: fp32 [B, k+1, V]; draft: fp32 [B, k, V]; drafts: int32 [B, k]; r: fp32
    [B, k] and u: fp32 [B] uniforms in [0, 1). Returns (n_accepted [B], next [B], errors).
    """
    lib = _load()
    target = np.ascontiguousarray(target, dtype=np.float32)
    B, k1, V = target.shape
    k = k1 - 1
    u = np.ascontiguousarray(u, dtype=np.float32)
    if k:
        draft = np.ascontiguousarray(draft, dtype=np.float32)
        drafts = np.ascontiguousarray(drafts, dtype=np.int32)
        r = np.ascontiguousarray(r, dtype=np.float32)
        assert draft.shape == (B, k, V) and drafts.shape == (B, k) and r.shape == (B, k)
    n = np.empty(B, np.int32)
    nxt = np.empty(B, np.int32)
    m = lib.kvo_sample_accept(B, k, V, _ptr(target), _ptr(draft), _ptr(drafts),
                              float(temperature), _ptr(r), _ptr(u), _ptr(n), _ptr(nxt))
    return n, nxt, _errs(m)
