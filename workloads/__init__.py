"""Seeded synthetic inputs for the KV-cached decoder step.

This package only draws random numbers and lays them out; it computes no part of
the decode method. Both the fp64 oracle (through the tests) and the CUDA library
(through the tests, ``bench.py`` and ``smoke()``) receive the exact arrays these
functions return, so the two sides always see bit-identical inputs.
"""

from .synth import (  # noqa: F401
    DTYPES,
    POISON,
    WORKLOADS,
    make_rng,
    normal_half,
    round_half_bits,
    gen_cache,
    gen_cache_device,
    gen_queries,
    gen_new_kv,
    gen_lens_uniform,
    gen_accept_inputs,
    gen_parents,
    gen_beam_select_inputs,
    gen_sample_inputs,
    seed_for,
)
