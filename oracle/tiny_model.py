"""Tiny fp64 decoder transformer for the end-to-end invariants -- TEST INFRASTRUCTURE ONLY.

A pre-LN decoder with the block structure of an encoder-decoder speech model:
token embedding plus a learned position table; per layer causal self-attention,
cross-attention over encoder frames, and an MLP; a final LayerNorm and an LM head.
Weights are random (drawn from the generator the caller passes); the invariants
below hold for any weights, which is the point the speculative-decoding pages make
about the method being model-agnostic ("실용적인 요점" of "추측 디코딩으로 Whisper 추론 속도
2배 향상").

Two independent ways to get logits:

* ``TinyDecoder.logits_full`` recomputes the whole sequence with numpy matrices and a
  causal mask, projecting the encoder K/V again on every call -- the "no cache"
  behaviour described in "自己回帰生成における計算の冗長性" of "nanoVLM における KV
  キャッシュ実装";
* ``CachedRunner.step`` feeds only the new tokens, appends their K/V with the
  oracle's ``kv_append`` and attends with the oracle's ``attention`` over the cache
  and over cross K/V projected once per window ("Inference 抽象と KV キャッシュ" of
  "Whisper のデコーダー内部：Beam Search、Logit フィルター、KV キャッシュ").

The decoding loops (plain greedy, speculative greedy with verify/accept/rollback,
beam search with cache reorder) are written from the same pages and only call the
oracle functions for the §8 operations.
"""

from __future__ import annotations

import numpy as np

from . import attention, beam_reorder, greedy_accept, kv_append


def _layer_norm(x, g, b, eps=1e-5):
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * g + b


def _softmax_last(s):
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


class TinyDecoder:
    def __init__(self, rng, vocab=64, d_model=64, n_heads=4, n_kv_heads=4, n_layers=2,
                 n_ctx=64, lm_gain=6.0):
        assert d_model % n_heads == 0 and n_heads % n_kv_heads == 0
        self.vocab, self.d, self.h, self.hkv = vocab, d_model, n_heads, n_kv_heads
        self.hd = d_model // n_heads
        self.n_layers, self.n_ctx = n_layers, n_ctx
        self.scale = 1.0 / np.sqrt(self.hd)
        d, hd = d_model, self.hd
        nrm = lambda *s, std=1.0: rng.standard_normal(size=s) * std  # noqa: E731
        self.embed = nrm(vocab, d, std=0.5)
        self.pos = nrm(n_ctx, d, std=0.1)
        self.layers = []
        for _ in range(n_layers):
            self.layers.append(dict(
                ln1=(1 + nrm(d, std=0.1), nrm(d, std=0.1)),
                wq=nrm(d, n_heads * hd, std=d ** -0.5),
                wk=nrm(d, n_kv_heads * hd, std=d ** -0.5),
                wv=nrm(d, n_kv_heads * hd, std=d ** -0.5),
                wo=nrm(n_heads * hd, d, std=(n_heads * hd) ** -0.5),
                ln2=(1 + nrm(d, std=0.1), nrm(d, std=0.1)),
                xq=nrm(d, n_heads * hd, std=d ** -0.5),
                xk=nrm(d, n_kv_heads * hd, std=d ** -0.5),
                xv=nrm(d, n_kv_heads * hd, std=d ** -0.5),
                xo=nrm(n_heads * hd, d, std=(n_heads * hd) ** -0.5),
                ln3=(1 + nrm(d, std=0.1), nrm(d, std=0.1)),
                w1=nrm(d, 4 * d, std=d ** -0.5),
                w2=nrm(4 * d, d, std=(4 * d) ** -0.5),
            ))
        self.lnf = (1 + nrm(d, std=0.1), nrm(d, std=0.1))
        self.lm = nrm(d, vocab, std=lm_gain * d ** -0.5)
        self.cross_calls = 0

    def perturbed(self, rng, noise: float):
        """A second model (the assistant) whose weights are this one's plus noise."""
        other = TinyDecoder.__new__(TinyDecoder)
        other.__dict__.update({k: v for k, v in self.__dict__.items()})
        jit = lambda a: a + rng.standard_normal(size=a.shape) * noise * np.std(a)  # noqa: E731
        other.embed = jit(self.embed)
        other.lm = jit(self.lm)
        other.layers = [{k: (tuple(jit(x) for x in v) if isinstance(v, tuple) else jit(v))
                         for k, v in lay.items()} for lay in self.layers]
        other.cross_calls = 0
        return other

    # -- cross-attention K/V of one audio window ---------------------------------------
    def project_cross(self, enc):
        """Per-layer cross K/V ``[Hkv, frames, hd]`` for one window's encoder output."""
        self.cross_calls += 1
        out = []
        for lay in self.layers:
            f = enc.shape[0]
            k = (enc @ lay["xk"]).reshape(f, self.hkv, self.hd).transpose(1, 0, 2)
            v = (enc @ lay["xv"]).reshape(f, self.hkv, self.hd).transpose(1, 0, 2)
            out.append((k, v))
        return out

    def _heads(self, x, w, n):
        B, T, _ = x.shape
        return (x @ w).reshape(B, T, n, self.hd).transpose(0, 2, 1, 3)  # [B, n, T, hd]

    def _expand(self, kv):
        """Repeat each KV head for its group of query heads."""
        return np.repeat(kv, self.h // self.hkv, axis=1)

    def _mlp(self, x, lay):
        h = _layer_norm(x, *lay["ln3"])
        return np.maximum(h @ lay["w1"], 0.0) @ lay["w2"]

    def _head(self, x):
        return _layer_norm(x, *self.lnf) @ self.lm

    # -- no cache: recompute everything --------------------------------------------------
    def logits_full(self, tokens, encs):
        """Logits ``[B, T, vocab]`` for ``tokens [B, T]``; ``encs[b]`` is row b's encoder output."""
        tokens = np.asarray(tokens)
        B, T = tokens.shape
        x = self.embed[tokens] + self.pos[np.arange(T)][None]
        cross = [self.project_cross(e) for e in encs]  # recomputed every call
        causal = np.triu(np.full((T, T), -np.inf), k=1)
        for li, lay in enumerate(self.layers):
            h = _layer_norm(x, *lay["ln1"])
            q = self._heads(h, lay["wq"], self.h)
            k = self._expand(self._heads(h, lay["wk"], self.hkv))
            v = self._expand(self._heads(h, lay["wv"], self.hkv))
            p = _softmax_last(np.einsum("bhqd,bhkd->bhqk", q, k) * self.scale + causal)
            o = np.einsum("bhqk,bhkd->bhqd", p, v).transpose(0, 2, 1, 3).reshape(B, T, -1)
            x = x + o @ lay["wo"]
            h = _layer_norm(x, *lay["ln2"])
            q = self._heads(h, lay["xq"], self.h)
            kx = np.stack([self._expand(c[li][0][None])[0] for c in cross])
            vx = np.stack([self._expand(c[li][1][None])[0] for c in cross])
            p = _softmax_last(np.einsum("bhqd,bhkd->bhqk", q, kx) * self.scale)
            o = np.einsum("bhqk,bhkd->bhqd", p, vx).transpose(0, 2, 1, 3).reshape(B, T, -1)
            x = x + o @ lay["xo"]
            x = x + self._mlp(x, lay)
        return self._head(x)


class CachedRunner:
    """Incremental decoding of ``model`` with per-layer caches ``[B, Hkv, cap, hd]``.

    Rows ``r`` share the cross K/V of window ``r // rows_per_window`` (beam rows of
    one audio window), projected once per window at construction.
    """

    def __init__(self, model: TinyDecoder, window_encs, rows_per_window: int = 1,
                 capacity: int | None = None):
        self.m = model
        self.rpw = rows_per_window
        self.B = len(window_encs) * rows_per_window
        self.cap = capacity or model.n_ctx
        shape = (self.B, model.hkv, self.cap, model.hd)
        self.K = [np.zeros(shape) for _ in range(model.n_layers)]
        self.V = [np.zeros(shape) for _ in range(model.n_layers)]
        self.lens = np.zeros(self.B, np.int32)
        per_window = [model.project_cross(e) for e in window_encs]
        self.frames = window_encs[0].shape[0]
        self.KX = [np.ascontiguousarray(np.stack([w[li][0] for w in per_window]))
                   for li in range(model.n_layers)]
        self.VX = [np.ascontiguousarray(np.stack([w[li][1] for w in per_window]))
                   for li in range(model.n_layers)]

    def step(self, new_tokens):
        """Feed ``new_tokens [B, q]`` (q >= 1) and return their logits ``[B, q, vocab]``."""
        m = self.m
        new_tokens = np.asarray(new_tokens)
        B, q = new_tokens.shape
        pos = self.lens[:, None] + np.arange(q)[None]
        x = m.embed[new_tokens] + m.pos[pos]
        lens_out = self.lens
        for li, lay in enumerate(m.layers):
            h = _layer_norm(x, *lay["ln1"])
            qh = np.ascontiguousarray(m._heads(h, lay["wq"], m.h))
            kn = np.ascontiguousarray(m._heads(h, lay["wk"], m.hkv))
            vn = np.ascontiguousarray(m._heads(h, lay["wv"], m.hkv))
            lens_out, err = kv_append(self.K[li], self.V[li], kn, vn, self.lens, "f64")
            assert not err
            o, err = attention(qh, self.K[li], self.V[li], "f64", lens=lens_out, causal=True,
                               scale=m.scale)
            assert not err
            x = x + o.transpose(0, 2, 1, 3).reshape(B, q, -1) @ lay["wo"]
            h = _layer_norm(x, *lay["ln2"])
            qx = np.ascontiguousarray(m._heads(h, lay["xq"], m.h))
            o, err = attention(qx, self.KX[li], self.VX[li], "f64", fixed_len=self.frames,
                               rows_per_kv=self.rpw, causal=False, scale=m.scale)
            assert not err
            x = x + o.transpose(0, 2, 1, 3).reshape(B, q, -1) @ lay["xo"]
            x = x + m._mlp(x, lay)
        self.lens = lens_out
        return m._head(x)

    def truncate(self, new_lens):
        """Roll the cache back to ``new_lens`` positions per row (metadata only)."""
        self.lens = np.asarray(new_lens, dtype=np.int32).copy()

    def reorder(self, parent, beam: int):
        """Gather every layer's K/V rows by ``parent`` (all rows share one length)."""
        assert np.all(self.lens == self.lens[0])
        L = int(self.lens[0])
        for li in range(self.m.n_layers):
            self.K[li], e1 = beam_reorder(self.K[li], parent, beam, L, "f64")
            self.V[li], e2 = beam_reorder(self.V[li], parent, beam, L, "f64")
            assert not e1 and not e2


# -- decoding loops ------------------------------------------------------------------------

def _argmax_f32(logits):
    return np.argmax(np.asarray(logits, dtype=np.float32), axis=-1)


def greedy_uncached(model, prompt, encs, n_new):
    toks = np.array(prompt)
    steps = []
    for _ in range(n_new):
        lg = model.logits_full(toks, encs)[:, -1]
        steps.append(lg)
        toks = np.concatenate([toks, _argmax_f32(lg)[:, None]], axis=1)
    return toks, steps


def greedy_cached(model, prompt, encs, n_new):
    """Prefill with the whole prompt, then one token per step."""
    run = CachedRunner(model, encs)
    toks = np.array(prompt)
    lg = run.step(toks)[:, -1]
    steps = [lg]
    toks = np.concatenate([toks, _argmax_f32(lg)[:, None]], axis=1)
    for _ in range(n_new - 1):
        lg = run.step(toks[:, -1:])[:, -1]
        steps.append(lg)
        toks = np.concatenate([toks, _argmax_f32(lg)[:, None]], axis=1)
    return toks, steps


def speculative_greedy(main, assistant, prompt, encs, n_new, k):
    """Greedy speculative decoding, batch 1: the assistant drafts ``k`` tokens, the main
    model verifies ``[last committed, d_0..d_{k-1}]`` in one causal block pass, the
    oracle accept keeps drafts up to the first mismatch plus the main model's token,
    and the main cache is truncated to the committed prefix.

    Returns ``(tokens, accepted_per_round)``.
    """
    prompt = np.array(prompt)
    assert prompt.shape[0] == 1
    seq = list(prompt[0])
    target = len(seq) + n_new
    mrun = CachedRunner(main, encs)
    arun = CachedRunner(assistant, encs)
    # Prime the main cache with all committed tokens but the last.
    if len(seq) > 1:
        mrun.step(np.array([seq[:-1]]))
    accepted = []
    while len(seq) < target:
        # assistant catches up on committed tokens it has not cached, then drafts k tokens
        have = int(arun.lens[0])
        lg = arun.step(np.array([seq[have:]]))[:, -1]
        drafts = []
        for i in range(k):
            d = int(_argmax_f32(lg)[0])
            drafts.append(d)
            if i + 1 < k:
                lg = arun.step(np.array([[d]]))[:, -1]
        T = len(seq)
        block = np.array([[seq[-1]] + drafts])
        logits = mrun.step(block).astype(np.float32)  # [1, k+1, vocab]
        n, nxt, _, _, err = greedy_accept(logits, np.array([drafts], np.int32))
        assert not err
        n = int(n[0])
        accepted.append(n)
        seq.extend(drafts[:n] + [int(nxt[0])])
        mrun.truncate([T + n])
        arun.truncate([T + min(n, k - 1)])
    return np.array([seq[:target]]), accepted


def _log_softmax(x):
    m = np.max(x, axis=-1, keepdims=True)
    return x - m - np.log(np.exp(x - m).sum(axis=-1, keepdims=True))


def _beam_select(logprobs, sums, beam):
    """One beam-search update for one window ("Inference 抽象と KV キャッシュ",
    BeamSearchDecoder): each beam offers its top beam+1 tokens, every continuation is
    scored by the summed log-probability, and the best ``beam`` are kept. Ties keep
    the lower (beam, rank) order. Returns (parents within the window, tokens, sums)."""
    cands = []
    for j in range(beam):
        order = np.argsort(-logprobs[j], kind="stable")[: beam + 1]
        for rank, tok in enumerate(order):
            cands.append((sums[j] + logprobs[j, tok], j, rank, int(tok)))
    cands.sort(key=lambda c: (-c[0], c[1], c[2]))
    best = cands[:beam]
    return (np.array([c[1] for c in best]), np.array([c[3] for c in best]),
            np.array([c[0] for c in best]))


def beam_search(model, prompt_row, window_encs, beam, n_steps, cached: bool):
    """Beam search over ``len(window_encs)`` windows, ``beam`` rows each, no EOT.

    ``cached=True`` runs the cache with ``reorder`` after each selection;
    ``cached=False`` recomputes every beam's full sequence each step.
    Returns ``(sequences [W*beam, T], scores [W*beam])``.
    """
    W = len(window_encs)
    R = W * beam
    seqs = np.tile(np.asarray(prompt_row)[None], (R, 1))
    sums = np.tile(np.r_[0.0, np.full(beam - 1, -np.inf)], W)  # only beam 0 is live at first
    row_encs = [window_encs[r // beam] for r in range(R)]
    run = CachedRunner(model, window_encs, rows_per_window=beam) if cached else None
    fed = 0
    for _ in range(n_steps):
        if cached:
            lg = run.step(seqs[:, fed:])[:, -1]
            fed = seqs.shape[1]
        else:
            lg = model.logits_full(seqs, row_encs)[:, -1]
        lp = _log_softmax(lg)
        parent = np.empty(R, np.int32)
        new_tok = np.empty(R, np.int64)
        new_sum = np.empty(R)
        for w in range(W):
            blk = slice(w * beam, (w + 1) * beam)
            p, t, s = _beam_select(lp[blk], sums[blk], beam)
            parent[blk] = w * beam + p
            new_tok[blk] = t
            new_sum[blk] = s
        if cached:
            run.reorder(parent, beam)
        seqs = np.concatenate([seqs[parent], new_tok[:, None]], axis=1)
        sums = new_sum
    return seqs, sums
