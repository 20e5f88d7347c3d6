"""Input recipe: named PRNG, shapes and value distributions of the decode workloads.

Every array is produced on the host from ``numpy.random.Generator(PCG64(seed))``.
Normals are drawn in fp64 and scaled, then rounded to the storage type:

* fp16: numpy's float64 -> float16 conversion (round to nearest, ties to even);
* bf16: float64 -> float32 (numpy, round to nearest even), then float32 -> bf16 by
  round-to-nearest-even on the float32 bit pattern.

16-bit storage types are returned as ``uint16`` bit patterns so that fp16 and bf16
travel the same way; ``dtype`` is the string ``"f16"`` or ``"bf16"``.

Cache positions at or beyond a row's length are filled with a NaN bit pattern
(``POISON``): a kernel that reads them into a result shows up as NaN.

Shapes (head_dim 64 throughout):

* tiny single layer: batch 1, 6 heads, self cache 32 cached + 1 new (capacity 33),
  cross K/V over 1500 encoder frames, fp16;
* Whisper-large-v2 shaped decoder step: 32 layers, batch 1, 20 heads, capacity 448
  (n_text_ctx), cross K/V 1500 frames per layer, fp16;
* speculative verify on those shapes: k = 5 drafts, vocabulary 51865, fp32 logits
  N(0, 2^2); each draft equals its row's argmax with probability 0.75, otherwise a
  uniformly drawn other id;
* GQA decoder LM: 30 layers, batch 16, 9 query heads over 3 KV heads, bf16, ragged
  lengths uniform in [256, 2048], capacity 2112, K stored already rotary-encoded;
* beam search: 8 audio windows x beam 5 = 40 rows, 32 layers, 20 heads, fp16,
  capacity 448, parents uniform inside each window's block of 5 rows;
* decode-attention sweep: batch {1,4,16,64} x length {128,512,2048,8192} x
  heads {20/20, 20/4};
* beam-search step selection: 8 audio windows x beam 5 = 40 rows of fp32 logits over
  a 51865-id vocabulary, N(0, 2^2); in 30% of the rows the EOT logit is set near the
  row's maximum (max + N(0, 0.5^2)) so that finished continuations occur; cumulative
  log-probabilities -U(0, 20) per row; a synthetic suppression set of 88 distinct ids
  and one blank id stand in for the tokenizer's lists (EOT is id 50257).

Q, K and V are N(0, 1) / 8 (i.e. 1/sqrt(head_dim)); the score scale is 1/8.
"""

from __future__ import annotations

import numpy as np

DTYPES = ("f16", "bf16")

# A quiet-NaN bit pattern per storage type, written to unused cache positions.
POISON = {"f16": np.uint16(0x7E00), "bf16": np.uint16(0x7FC0)}

WORKLOADS = {
    "tiny_layer": dict(
        n_layers=1, batch=1, n_q_heads=6, n_kv_heads=6, head_dim=64, dtype="f16",
        cached=32, new=1, capacity=33, cross_len=1500, qkv_std=0.125, scale=0.125,
    ),
    "whisper_large_v2_step": dict(
        n_layers=32, batch=1, n_q_heads=20, n_kv_heads=20, head_dim=64, dtype="f16",
        capacity=448, cross_len=1500, qkv_std=0.125, scale=0.125, len_range=(1, 447),
    ),
    "whisper_verify": dict(
        n_layers=32, batch=1, n_q_heads=20, n_kv_heads=20, head_dim=64, dtype="f16",
        capacity=448, cross_len=1500, qkv_std=0.125, scale=0.125, k=5, vocab=51865,
        logit_std=2.0, p_match=0.75, len_range=(0, 443),
    ),
    "gqa_lm_step": dict(
        n_layers=30, batch=16, n_q_heads=9, n_kv_heads=3, head_dim=64, dtype="bf16",
        capacity=2112, len_lo=256, len_hi=2048, qkv_std=0.125, scale=0.125,
    ),
    "beam_step": dict(
        n_layers=32, windows=8, beam=5, n_q_heads=20, n_kv_heads=20, head_dim=64,
        dtype="f16", capacity=448, cross_len=1500, lens=(32, 224, 440),
        qkv_std=0.125, scale=0.125,
    ),
    "beam_select": dict(
        windows=8, beam=5, vocab=51865, logit_std=2.0, p_eot=0.3, eot=50257,
        n_suppress=88, blank=(220,), cum_range=(0.0, 20.0),
    ),
    "decode_sweep": dict(
        batches=(1, 4, 16, 64), lens=(128, 512, 2048, 8192),
        heads=((20, 20), (20, 4)), head_dim=64, dtype="f16", qkv_std=0.125, scale=0.125,
    ),
}

_WORKLOAD_IDS = {name: i + 1 for i, name in enumerate(WORKLOADS)}


def seed_for(workload: str, layer: int = 0, salt: int = 0) -> int:
    """Fixed seed per workload and layer: 1000 * workload id + layer (+ salt)."""
    return 1000 * _WORKLOAD_IDS[workload] + layer + 100_000 * salt


def make_rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    bits = x32.view(np.uint32).astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def round_half_bits(x, dtype: str) -> np.ndarray:
    """fp64 values rounded to fp16/bf16 (nearest even), returned as uint16 bits."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return _f32_to_bf16_bits(x.astype(np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


def normal_half(rng: np.random.Generator, shape, std: float, dtype: str) -> np.ndarray:
    """N(0, std^2) drawn in fp64, rounded to fp16/bf16, returned as uint16 bits."""
    return round_half_bits(rng.standard_normal(size=shape) * std, dtype)


def gen_cache(rng, batch: int, n_kv_heads: int, capacity: int, head_dim: int,
              dtype: str, std: float, lens=None):
    """K and V caches ``[batch, n_kv_heads, capacity, head_dim]`` (uint16 bits).

    Positions ``t >= lens[b]`` hold ``POISON``; ``lens=None`` fills every position.
    """
    shape = (batch, n_kv_heads, capacity, head_dim)
    k = normal_half(rng, shape, std, dtype)
    v = normal_half(rng, shape, std, dtype)
    if lens is not None:
        lens = np.asarray(lens, dtype=np.int64).reshape(batch)
        pos = np.arange(capacity)[None, :]
        dead = pos >= lens[:, None]  # [batch, capacity]
        k[dead[:, None, :, None].repeat(n_kv_heads, 1).repeat(head_dim, 3)] = POISON[dtype]
        v[dead[:, None, :, None].repeat(n_kv_heads, 1).repeat(head_dim, 3)] = POISON[dtype]
    return k, v


def gen_queries(rng, batch: int, n_q_heads: int, qlen: int, head_dim: int,
                dtype: str, std: float) -> np.ndarray:
    """Query block ``[batch, n_q_heads, qlen, head_dim]`` (uint16 bits)."""
    return normal_half(rng, (batch, n_q_heads, qlen, head_dim), std, dtype)


def gen_new_kv(rng, batch: int, n_kv_heads: int, q: int, head_dim: int,
               dtype: str, std: float):
    """New tokens' K and V ``[batch, n_kv_heads, q, head_dim]`` (uint16 bits)."""
    shape = (batch, n_kv_heads, q, head_dim)
    return normal_half(rng, shape, std, dtype), normal_half(rng, shape, std, dtype)


def gen_lens_uniform(rng, batch: int, lo: int, hi: int) -> np.ndarray:
    """Ragged lengths, uniform integers in ``[lo, hi]`` (int32)."""
    return rng.integers(lo, hi + 1, size=batch).astype(np.int32)


def gen_accept_inputs(rng, batch: int, k: int, vocab: int, logit_std: float = 2.0,
                      p_match: float = 0.75):
    """Main-model logits ``[batch, k+1, vocab]`` fp32 and drafts ``[batch, k]`` int32.

    Logits are N(0, logit_std^2) rounded to fp32. Draft ``i`` is the position of
    row ``i``'s largest logit with probability ``p_match`` (independently per i),
    otherwise a uniformly drawn different id. ``numpy.argmax`` is used here only
    to build the drafts; no expected value is derived from it.
    """
    logits = (rng.standard_normal(size=(batch, k + 1, vocab)) * logit_std).astype(np.float32)
    top = np.argmax(logits[:, :k, :], axis=-1)  # [batch, k]
    match = rng.random(size=(batch, k)) < p_match
    other = rng.integers(0, vocab - 1, size=(batch, k))
    other = other + (other >= top)  # uniform over the vocab minus the top id
    drafts = np.where(match, top, other).astype(np.int32)
    return logits, drafts


def gen_parents(rng, windows: int, beam: int) -> np.ndarray:
    """Beam parents ``[windows*beam]`` int32, uniform inside each window's block."""
    base = np.repeat(np.arange(windows) * beam, beam)
    return (base + rng.integers(0, beam, size=windows * beam)).astype(np.int32)


def gen_beam_select_inputs(rng, windows: int, beam: int, vocab: int, *, logit_std: float = 2.0,
                           p_eot: float = 0.3, eot: int = 50257, n_suppress: int = 88,
                           cum_range=(0.0, 20.0)):
    """Inputs of one beam-search selection step.

    Returns ``(logits [windows*beam, vocab] fp32, cum [windows*beam] fp32,
    suppress [n_suppress] int32)``. Logits are N(0, logit_std^2); with probability
    ``p_eot`` a row's EOT logit is replaced by the row's maximum plus N(0, 0.5^2).
    ``cum`` is -U(cum_range). ``suppress`` holds distinct ids drawn uniformly from the
    vocabulary without EOT.
    """
    rows = windows * beam
    logits = (rng.standard_normal(size=(rows, vocab)) * logit_std).astype(np.float32)
    hit = rng.random(size=rows) < p_eot
    bump = (logits.max(axis=1) + rng.standard_normal(size=rows) * 0.5).astype(np.float32)
    if 0 <= eot < vocab:
        logits[hit, eot] = bump[hit]
    cum = (-rng.uniform(cum_range[0], cum_range[1], size=rows)).astype(np.float32)
    pool = np.array([v for v in range(vocab) if v != eot]) if vocab < 4096 else None
    if pool is None:
        sup = rng.choice(vocab, size=n_suppress + 1, replace=False)
        sup = sup[sup != eot][:n_suppress]
    else:
        sup = rng.choice(pool, size=min(n_suppress, pool.size), replace=False)
    return logits, cum, np.sort(sup).astype(np.int32)


def gen_sample_inputs(rng, batch: int, k: int, vocab: int, *, logit_std: float = 2.0,
                      draft_noise: float = 1.0, p_match: float = 0.75):
    """Inputs of temperature sampling / stochastic speculative acceptance.

    Returns ``(target [batch, k+1, vocab] fp32, draft [batch, k, vocab] fp32, drafts
    [batch, k] int32, r [batch, k] fp32, u [batch] fp32)``. The draft logits are the
    target logits plus N(0, draft_noise^2); draft i is the draft row's largest logit with
    probability p_match, else a uniform id. ``numpy.argmax`` only builds the drafts.
    """
    target = (rng.standard_normal(size=(batch, k + 1, vocab)) * logit_std).astype(np.float32)
    noise = (rng.standard_normal(size=(batch, k, vocab)) * draft_noise).astype(np.float32)
    draft = (target[:, :k] + noise).astype(np.float32)
    top = np.argmax(draft, axis=-1) if k else np.zeros((batch, 0), np.int64)
    match = rng.random(size=(batch, k)) < p_match
    other = rng.integers(0, vocab, size=(batch, k))
    drafts = np.where(match, top, other).astype(np.int32)
    r = rng.random(size=(batch, k)).astype(np.float32)
    u = rng.random(size=batch).astype(np.float32)
    return target, draft, drafts, r, u


def gen_cache_device(seed: int, batch: int, n_kv_heads: int, capacity: int, head_dim: int,
                     dtype: str, std: float, device="cuda"):
    """Full-size K and V caches ``[batch, n_kv_heads, capacity, head_dim]`` drawn on the
    device: torch's seeded Philox generator on ``device``, N(0, std^2) rounded by torch to
    fp16/bf16. For caches too large to draw on the host in reasonable time (gigabytes);
    a test copies the rows it checks back to the host, so both sides see the same bits.
    Returns two torch tensors (the caller keeps them alive)."""
    import torch

    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (batch, n_kv_heads, capacity, head_dim)
    k = torch.empty(shape, dtype=tdt, device=device).normal_(0.0, std, generator=gen)
    v = torch.empty(shape, dtype=tdt, device=device).normal_(0.0, std, generator=gen)
    return k, v
