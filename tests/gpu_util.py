"""Helpers for the GPU parity tests: host<->device copies of the seeded inputs and the
attention tolerance. The attention bar is max-abs error <= 1e-2 and relative Frobenius
error <= 5e-3 against the fp64 oracle; integer and copy results must be bit-exact."""

import numpy as np
import pytest
import torch

MAX_ABS = 1e-2
REL_FRO = 5e-3
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from kv_cached_decode_gb300 import build, load_library

    build.build()
    load_library()


def dev16(bits: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(TORCH_DT[dtype]).cuda()


def host16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def dev_i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attn_errors(got_bits, want, dtype):
    g = f64(got_bits, dtype)
    diff = g - want
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    nrm = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(diff)) / nrm if nrm > 0 else float(np.linalg.norm(diff))
    return max_abs, rel


def assert_attn_close(got_bits, want, dtype, what=""):
    assert np.all(np.isfinite(f64(got_bits, dtype))), f"non-finite output {what}"
    max_abs, rel = attn_errors(got_bits, want, dtype)
    assert max_abs <= MAX_ABS and rel <= REL_FRO, f"{what}: max_abs={max_abs:.3e} rel={rel:.3e}"


def new_err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")
