"""Python binding of ``libkvdecode.so`` -- the GB300 KV-cached decoder-step library.

Argument marshalling only: every function passes ``torch.Tensor.data_ptr()`` values,
sizes and the current CUDA stream to the C entry point of the same name declared in
``include/kvdecode.h``; all work happens in the library's CUDA kernels. There is no
fallback: if the library has not been built (``python -m kv_cached_decode_gb300.build``)
or a call fails, an exception is raised.

Tensors: caches are ``[batch, n_kv_heads, capacity, 64]`` fp16/bf16 CUDA tensors with
the last axis contiguous; queries/outputs are contiguous ``[batch, n_q_heads, qlen, 64]``;
lengths, drafts, parents and outputs of ``kvd_greedy_accept`` are int32 CUDA tensors;
logits are contiguous fp32 ``[batch, k+1, vocab]`` (``kvd_greedy_accept``) or
``[windows*beam, vocab]`` (``kvd_beam_select``).
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvdecode.so")

KVD_OK = 0
STATUS_NAMES = {0: "KVD_OK", 1: "KVD_ERR_INVALID_ARG", 2: "KVD_ERR_UNSUPPORTED",
                3: "KVD_ERR_WORKSPACE", 4: "KVD_ERR_CUDA", 16: "KVD_ERR_LEN_OVERFLOW",
                17: "KVD_ERR_BAD_INDEX", 18: "KVD_ERR_BAD_TOKEN", 19: "KVD_ERR_NAN",
                20: "KVD_ERR_TIMEOUT"}
KVD_F16, KVD_BF16 = 0, 1
KVD_OP_DECODE_ATTN, KVD_OP_VERIFY_ATTN, KVD_OP_GREEDY_ACCEPT, KVD_OP_SAMPLE_ACCEPT = 0, 1, 2, 3
KVD_FLAG_PDL, KVD_FLAG_EARLY_KV = 1, 2
KVD_FLAG_TEST_STALL = 1 << 8  # test only: see include/kvdecode.h
KVD_WS_COUNTER_BYTES = 65536
HEAD_DIM = 64

EXPORTED = ("kvd_kv_append", "kvd_decode_attn", "kvd_verify_attn", "kvd_greedy_accept",
            "kvd_beam_reorder_kv", "kvd_workspace_size", "kvd_status_string", "kvd_version",
            "kvd_decode_attn_noalloc", "kvd_prefill_attn", "kvd_rope", "kvd_beam_select",
            "kvd_kv_append_rope", "kvd_sample_accept", "kvd_noalloc_test_fill_counters")


class KvdError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call} failed: {STATUS_NAMES.get(status, status)}")


class Cache(ctypes.Structure):
    """Mirror of ``kvd_cache``: one layer's K and V buffers with shared strides."""

    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64),
                ("stride_t", ctypes.c_int64), ("batch", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("capacity", ctypes.c_int32)]


class NewTokens(ctypes.Structure):
    """Mirror of ``kvd_new_tokens``: new K/V appended inside an attention call."""

    _fields_ = [("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("lens_out", ctypes.c_void_p), ("rope_base", ctypes.c_float)]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load the CUDA library (raises if it was never built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m kv_cached_decode_gb300.build` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        P, I32, U32, F, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float,
                              ctypes.c_size_t)
        CP = ctypes.POINTER(Cache)
        NP = ctypes.POINTER(NewTokens)
        sig = {
            "kvd_kv_append": [I32, CP, I32, I32, P, P, P, P, U32, P, P],
            "kvd_decode_attn": [I32, I32, I32, P, CP, P, I32, NP, I32, F, P, P, SZ, U32, P, P],
            "kvd_decode_attn_noalloc": [I32, I32, I32, P, CP, P, I32, NP, I32, F, P, U32, P, P],
            "kvd_noalloc_test_fill_counters": [ctypes.c_uint8, P],
            "kvd_verify_attn": [I32, I32, I32, I32, P, CP, P, I32, NP, I32, I32, F, P, P, SZ,
                                U32, P, P],
            "kvd_prefill_attn": [I32, I32, I32, I32, P, CP, P, P, P, P, P, F, F, P, U32, P, P],
            "kvd_kv_append_rope": [I32, CP, I32, I32, P, P, P, P, F, U32, P, P],
            "kvd_sample_accept": [P, P, P, I32, I32, I32, F, P, P, P, P, P, SZ, U32, P, P],
            "kvd_rope": [I32, I32, I32, P, I32, P, I32, P, F, U32, P, P],
            "kvd_greedy_accept": [P, I32, I32, I32, P, P, P, P, P, P, SZ, U32, P, P],
            "kvd_beam_reorder_kv": [I32, CP, I32, I32, I32, P, P, I32, U32, P, P],
            "kvd_beam_select": [P, I32, I32, I32, P, P, I32, P, I32, I32, I32, P, P, P, P, P,
                                P, P, P, U32, P, P],
            "kvd_workspace_size": [I32, I32, I32, I32, I32, I32, I32, I32],
            "kvd_status_string": [I32],
            "kvd_version": [],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = I32
        lib.kvd_workspace_size.restype = SZ
        lib.kvd_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return KVD_F16
    if t.dtype == torch.bfloat16:
        return KVD_BF16
    raise TypeError(f"expected float16 or bfloat16, got {t.dtype}")


_I32, _F32 = torch.int32, torch.float32


def _ptr(t, dtype=None, what="tensor"):
    """The device address of a contiguous CUDA tensor (None stays None). Anything else is
    refused here: the library would read a host address or a strided view as a dense
    device array."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _dev(t, what):
    return _ptr(t, None, what)


def _i32(t, what):
    return _ptr(t, _I32, what)


def _f32(t, what):
    return _ptr(t, _F32, what)


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _append_arg(append):
    """``append`` is None or ``(k_new, v_new, lens_out_or_None[, rope_base])``: device
    tensors, and the rotary base (0 or absent: no rotation)."""
    if append is None:
        return None
    k_new, v_new, lens_out = append[:3]
    rope_base = float(append[3]) if len(append) > 3 else 0.0
    kp, vp = _dev(k_new, "k_new"), _dev(v_new, "v_new")
    lp = _i32(lens_out, "lens_out")
    return ctypes.byref(NewTokens(kp.value, vp.value, None if lp is None else lp.value,
                                  rope_base))


def _check(status: int, call: str):
    if status != KVD_OK:
        raise KvdError(status, call)


def make_cache(k: torch.Tensor, v: torch.Tensor) -> Cache:
    """Describe one layer's ``[batch, heads, capacity, 64]`` K/V tensors for the C ABI."""
    if k.shape != v.shape or k.stride() != v.stride() or k.dtype != v.dtype:
        raise ValueError("K and V must share shape, strides and dtype")
    if k.dim() != 4 or k.shape[3] != HEAD_DIM or k.stride(3) != 1:
        raise ValueError("cache must be [batch, heads, capacity, 64] with the last axis contiguous")
    if not (k.is_cuda and v.is_cuda):
        raise ValueError("cache tensors must be CUDA tensors")
    B, H, cap, D = k.shape
    c = Cache(k.data_ptr(), v.data_ptr(), k.stride(0), k.stride(1), k.stride(2), B, H, D, cap)
    c._tensors = (k, v)  # the struct holds raw pointers: keep the tensors alive with it
    return c


def kvd_version() -> int:
    return load_library().kvd_version()


def kvd_status_string(status: int) -> str:
    return load_library().kvd_status_string(status).decode()


def kvd_workspace_size(op: int, batch: int, n_q_heads: int = 1, n_kv_heads: int = 1,
                       rows_per_kv: int = 1, qlen: int = 1, max_len: int = 0,
                       vocab: int = 0) -> int:
    return load_library().kvd_workspace_size(op, batch, n_q_heads, n_kv_heads, rows_per_kv, qlen,
                                             max_len, vocab)


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled device workspace (the counter region must start at zero)."""
    return torch.zeros(max(int(nbytes), KVD_WS_COUNTER_BYTES), dtype=torch.uint8,
                       device=device or "cuda")


def kvd_kv_append(cache: Cache, k_new, v_new, lens_in, lens_out=None, flags: int = 0,
                  dev_err=None, stream=None):
    B, H, q, D = k_new.shape
    _check(load_library().kvd_kv_append(_dtype_code(k_new), ctypes.byref(cache), B, q,
                                        _dev(k_new, "k_new"), _dev(v_new, "v_new"),
                                        _i32(lens_in, "lens_in"), _i32(lens_out, "lens_out"), flags,
                                        _i32(dev_err, "dev_err"), _stream(stream)), "kvd_kv_append")


def kvd_kv_append_rope(cache: Cache, k_new, v_new, lens_in, lens_out=None,
                       rope_base: float = 10000.0, flags: int = 0, dev_err=None, stream=None):
    B, H, q, D = k_new.shape
    _check(load_library().kvd_kv_append_rope(_dtype_code(k_new), ctypes.byref(cache), B, q,
                                             _dev(k_new, "k_new"), _dev(v_new, "v_new"),
                                             _i32(lens_in, "lens_in"), _i32(lens_out, "lens_out"),
                                             rope_base, flags, _i32(dev_err, "dev_err"),
                                             _stream(stream)), "kvd_kv_append_rope")


def kvd_decode_attn(q, cache: Cache, out, workspace, lens=None, fixed_len: int = 0,
                    rows_per_kv: int = 1, scale: float = 0.125, flags: int = 0,
                    dev_err=None, stream=None, append=None):
    B, Hq, ql, D = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().kvd_decode_attn(_dtype_code(q), B, Hq, _dev(q, "q"), ctypes.byref(cache),
                                          _i32(lens, "lens"), fixed_len, _append_arg(append),
                                          rows_per_kv, scale, _dev(out, "out"),
                                          _dev(workspace, "workspace"), ws_bytes, flags,
                                          _i32(dev_err, "dev_err"), _stream(stream)),
           "kvd_decode_attn")


def kvd_decode_attn_noalloc(q, cache: Cache, out, lens=None, fixed_len: int = 0,
                            rows_per_kv: int = 1, scale: float = 0.125, flags: int = 0,
                            dev_err=None, stream=None, append=None):
    """kvd_decode_attn without a workspace: the library's built-in scratch is used."""
    B, Hq, ql, D = q.shape
    _check(load_library().kvd_decode_attn_noalloc(_dtype_code(q), B, Hq, _dev(q, "q"),
                                                  ctypes.byref(cache), _i32(lens, "lens"),
                                                  fixed_len, _append_arg(append), rows_per_kv,
                                                  scale, _dev(out, "out"), flags,
                                                  _i32(dev_err, "dev_err"), _stream(stream)),
           "kvd_decode_attn_noalloc")


def kvd_noalloc_test_fill_counters(byte_value: int, stream=None):
    """Test support: fill the built-in scratch's arrival counters with ``byte_value``."""
    _check(load_library().kvd_noalloc_test_fill_counters(byte_value, _stream(stream)),
           "kvd_noalloc_test_fill_counters")


def kvd_verify_attn(q, cache: Cache, out, workspace, lens=None, fixed_len: int = 0,
                    rows_per_kv: int = 1, causal: bool = True, scale: float = 0.125,
                    flags: int = 0, dev_err=None, stream=None, append=None):
    B, Hq, ql, D = q.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load_library().kvd_verify_attn(_dtype_code(q), B, Hq, ql, _dev(q, "q"),
                                          ctypes.byref(cache), _i32(lens, "lens"), fixed_len,
                                          _append_arg(append), rows_per_kv, int(bool(causal)),
                                          scale, _dev(out, "out"), _dev(workspace, "workspace"),
                                          ws_bytes, flags, _i32(dev_err, "dev_err"),
                                          _stream(stream)), "kvd_verify_attn")


def kvd_prefill_attn(q, cache: Cache, k_new, v_new, plens, out, lens_in=None, lens_out=None,
                     scale: float = 0.125, rope_base: float = 0.0, flags: int = 0,
                     dev_err=None, stream=None):
    """Prefill: append the prompt's K/V (rows j < plens[b]) and run causal attention of
    the prompt. q, out: [batch, n_q_heads, max_len, 64]; k_new, v_new: [batch,
    n_kv_heads, max_len, 64]. rope_base > 0: rotary encoding of the prompt."""
    B, Hq, T, D = q.shape
    _check(load_library().kvd_prefill_attn(_dtype_code(q), B, Hq, T, _dev(q, "q"),
                                           ctypes.byref(cache), _dev(k_new, "k_new"),
                                           _dev(v_new, "v_new"), _i32(lens_in, "lens_in"),
                                           _i32(plens, "plens"), _i32(lens_out, "lens_out"), scale,
                                           rope_base, _dev(out, "out"), flags,
                                           _i32(dev_err, "dev_err"), _stream(stream)),
           "kvd_prefill_attn")


def kvd_rope(q=None, k=None, pos0=None, base: float = 10000.0, flags: int = 0, dev_err=None,
             stream=None):
    """Rotary encoding, in place, of q [batch, n_q_heads, n, 64] and/or k [batch,
    n_k_heads, n, 64]; token j of row b at position pos0[b] + j."""
    ref = q if q is not None else k
    B, _, n, _ = ref.shape
    _check(load_library().kvd_rope(_dtype_code(ref), B, n, _dev(q, "q"),
                                   0 if q is None else q.shape[1], _dev(k, "k"),
                                   0 if k is None else k.shape[1], _i32(pos0, "pos0"), base, flags,
                                   _i32(dev_err, "dev_err"), _stream(stream)), "kvd_rope")


def kvd_greedy_accept(logits, draft, n_accepted, next_token, workspace, n_min=None,
                      argmax=None, flags: int = 0, dev_err=None, stream=None):
    B, k1, V = logits.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load_library().kvd_greedy_accept(_f32(logits, "logits"), B, k1 - 1, V,
                                            _i32(draft, "draft"), _i32(n_accepted, "n_accepted"),
                                            _i32(next_token, "next_token"), _i32(n_min, "n_min"),
                                            _i32(argmax, "argmax"), _dev(workspace, "workspace"),
                                            ws_bytes, flags, _i32(dev_err, "dev_err"),
                                            _stream(stream)), "kvd_greedy_accept")


def kvd_beam_reorder_kv(caches, rows: int, beam: int, parent, lens=None, fixed_len: int = 0,
                        dtype=torch.float16, flags: int = 0, dev_err=None, stream=None):
    arr = (Cache * len(caches))(*caches)
    code = KVD_F16 if dtype == torch.float16 else KVD_BF16
    _check(load_library().kvd_beam_reorder_kv(code, arr, len(caches), rows, beam,
                                              _i32(parent, "parent"), _i32(lens, "lens"), fixed_len,
                                              flags, _i32(dev_err, "dev_err"), _stream(stream)),
           "kvd_beam_reorder_kv")


def kvd_beam_select(logits, beam: int, *, cum=None, suppress=None, blank=None,
                    eot: int = 0, first_step: bool = False, row_token=None, row_logprob=None,
                    parent=None, token=None, new_cum=None, n_finished=None, fin_parent=None,
                    fin_score=None, flags: int = 0, dev_err=None, stream=None):
    """Logit filters + one beam-search selection step over ``logits [windows*beam, V]``.

    ``suppress``/``blank`` are int32 CUDA tensors of ids; the walk outputs (``parent``
    ... ``fin_score``) are all given or all None.
    """
    rows, V = logits.shape
    n_sup = 0 if suppress is None else suppress.numel()
    n_blank = 0 if blank is None else blank.numel()
    _check(load_library().kvd_beam_select(_f32(logits, "logits"), rows // beam, beam, V,
                                          _f32(cum, "cum"), _i32(suppress, "suppress"), n_sup,
                                          _i32(blank, "blank"), n_blank, eot, int(bool(first_step)),
                                          _i32(row_token, "row_token"),
                                          _f32(row_logprob, "row_logprob"), _i32(parent, "parent"),
                                          _i32(token, "token"), _f32(new_cum, "new_cum"),
                                          _i32(n_finished, "n_finished"),
                                          _i32(fin_parent, "fin_parent"),
                                          _f32(fin_score, "fin_score"), flags,
                                          _i32(dev_err, "dev_err"), _stream(stream)),
           "kvd_beam_select")


def kvd_sample_accept(target, u, n_accepted, next_token, workspace, temperature: float = 1.0,
                      draft=None, drafts=None, r=None, flags: int = 0, dev_err=None,
                      stream=None):
    """Temperature sampling (target [B, 1, V]) or stochastic speculative acceptance of k
    drafts (target [B, k+1, V], draft [B, k, V], drafts and r [B, k]); u: [B] uniforms;
    workspace: kvd_workspace_size(KVD_OP_SAMPLE_ACCEPT, B, qlen=k, vocab=V) bytes."""
    B, k1, V = target.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(load_library().kvd_sample_accept(_f32(target, "target"), _f32(draft, "draft"),
                                            _i32(drafts, "drafts"), B, k1 - 1, V, temperature,
                                            _f32(r, "r"), _f32(u, "u"),
                                            _i32(n_accepted, "n_accepted"),
                                            _i32(next_token, "next_token"),
                                            _dev(workspace, "workspace"), ws_bytes, flags,
                                            _i32(dev_err, "dev_err"), _stream(stream)),
           "kvd_sample_accept")
