"""The timed decoder step itself against the fp64 oracle.

bench.py times one CUDA graph of the Whisper-shaped step: per layer, a self decode with
the new token appended in the same launch, a cross decode over 1500 frames, a causal
5-token verify with its block appended, and a verify over the cross frames, all with PDL
and early K/V staging; then one greedy accept over [6, 51865]. This test builds that
step with bench.py's own class and launch flags, captures and replays the graph, and
checks sampled layers' outputs (every head, all four calls) and the accept result
against the oracle. The oracle's inputs come from the host generators only: the caches
are regenerated from their seeds, the new tokens and queries are read from the packed
host buffer the step uploads. Tolerance: max-abs 1e-2, rel-Frobenius 5e-3 (accept:
bit-exact).
"""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_attn_close, host16, require_gpu
from workloads import gen_cache, make_rng, seed_for

pytestmark = pytest.mark.gpu
D = 64


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_whisper_step_as_timed_matches_oracle():
    import bench
    import kv_cached_decode_gb300 as kvd

    dev = torch.device("cuda:0")
    step = bench.WhisperStep(dev, flags=kvd.KVD_FLAG_PDL,
                             cross_flags=kvd.KVD_FLAG_PDL | kvd.KVD_FLAG_EARLY_KV, fused=True)
    stream = torch.cuda.Stream(device=dev)
    g = bench.capture(torch, step.run, stream)  # one eager pass, then the graph
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    assert step.err.item() == 0
    assert step.dec_lens.item() == step.Ld + 1 and step.ver_lens.item() == step.Lv + step.k

    H, cap, F, k, NL = step.H, step.cap, step.F, step.k, step.NL
    qd, qv = H * D, H * k * D
    per_layer = 4 * qd + 4 * qv
    halves = step.h_in.numpy()[: step.n_halves].view(np.uint16)

    def part(layer, off, size, shape):
        base = layer * per_layer + off
        return halves[base: base + size].reshape(shape).copy()

    for layer in (0, 13, NL - 1):
        q_self = part(layer, 0, qd, (1, H, 1, D))
        q_cross = part(layer, qd, qd, (1, H, 1, D))
        kn1 = part(layer, 2 * qd, qd, (1, H, 1, D))
        vn1 = part(layer, 3 * qd, qd, (1, H, 1, D))
        qv_self = part(layer, 4 * qd, qv, (1, H, k, D))
        qv_cross = part(layer, 4 * qd + qv, qv, (1, H, k, D))
        kn5 = part(layer, 4 * qd + 2 * qv, qv, (1, H, k, D))
        vn5 = part(layer, 4 * qd + 3 * qv, qv, (1, H, k, D))
        rng = make_rng(seed_for("whisper_large_v2_step", layer, 0))
        K, V = gen_cache(rng, 1, H, cap, D, "f16", 0.125, lens=[step.Ld])
        Kx, Vx = gen_cache(rng, 1, H, F, D, "f16", 0.125)
        rng = make_rng(seed_for("whisper_verify", layer, 0))
        Kv, Vv = gen_cache(rng, 1, H, cap, D, "f16", 0.125, lens=[step.Lv])
        Kvx, Vvx = gen_cache(rng, 1, H, F, D, "f16", 0.125)
        # decode: append the new token at 447, attend over 448 and over the 1500 frames
        lo, _ = oracle.kv_append(K, V, kn1, vn1, np.array([step.Ld], np.int32), "f16")
        w_self, _ = oracle.attention(q_self, K, V, "f16", lens=lo)
        w_cross, _ = oracle.attention(q_cross, Kx, Vx, "f16", fixed_len=F)
        # verify: append the 5-token block at 443, causal over 448, then the cross frames
        lo5, _ = oracle.kv_append(Kv, Vv, kn5, vn5, np.array([step.Lv], np.int32), "f16")
        w_vself, _ = oracle.attention(qv_self, Kv, Vv, "f16", lens=lo5, causal=True)
        w_vcross, _ = oracle.attention(qv_cross, Kvx, Vvx, "f16", fixed_len=F)
        assert_attn_close(host16(step.o_self[layer]), w_self, "f16", f"layer {layer} self")
        assert_attn_close(host16(step.o_cross[layer]), w_cross, "f16", f"layer {layer} cross")
        assert_attn_close(host16(step.ov_self[layer]), w_vself, "f16", f"layer {layer} verify")
        assert_attn_close(host16(step.ov_cross[layer]), w_vcross, "f16",
                          f"layer {layer} verify cross")
        # the appended rows landed in the device caches
        assert np.array_equal(host16(step.dec_self[layer][0])[:, :, : step.Ld + 1],
                              K[:, :, : step.Ld + 1])
        assert np.array_equal(host16(step.ver_self[layer][1])[:, :, : step.Lv + k],
                              Vv[:, :, : step.Lv + k])
    n, nxt, _, _, _ = oracle.greedy_accept(step.host_logits, step.host_draft)
    assert int(step.n_acc.item()) == int(n[0]) and int(step.next_tok.item()) == int(nxt[0])
