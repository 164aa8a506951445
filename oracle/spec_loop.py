"""Speculative-decoding loop on a tiny random causal target -- TEST
INFRASTRUCTURE ONLY (CPU, float64).

Used to pin the oracle's verify-accept and loop semantics to the property
the pages promise: speculative decoding is lossless, i.e. under greedy
decoding it emits exactly the target's own greedy stream ([P1] overview
table "lossless" speedup; [P2] "DFlash는 손실 없는 가속을 보장한다" paragraph).

Loop order follows [P1] "추론 구조": target prefill taps a fixed set of
layers spread from shallow to deep, the fused feature is injected into every
drafter layer's KV cache and reused, the drafter decodes the masked block in
one pass, the target verifies the block in parallel.
"""
from __future__ import annotations

import numpy as np

from . import dflash_ref as ref


def tap_layers(n_layers: int, n_taps: int = 5) -> list[int]:
    """1-indexed target layers whose outputs are tapped: spread evenly from
    the second layer to the third-from-last ([P1] 실험 설정 table, "타깃
    hidden feature" row; [P4] §3.1)."""
    return [int(round(x)) for x in np.linspace(2, n_layers - 2, n_taps)]


class TinyTarget:
    """A small pre-norm causal transformer with random weights (float64).
    Only its greedy behaviour and its hidden states matter here."""

    def __init__(self, seed=7, vocab=64, d=64, n_layers=8, n_heads=2, d_ffn=128):
        rng = np.random.default_rng(seed)
        self.V, self.d, self.L, self.H = vocab, d, n_layers, n_heads
        self.dh = d // n_heads
        self.embed = rng.standard_normal((vocab, d))
        self.layers = []
        for _ in range(n_layers):
            self.layers.append({
                "wq": rng.standard_normal((d, d)) / np.sqrt(d),
                "wk": rng.standard_normal((d, d)) / np.sqrt(d),
                "wv": rng.standard_normal((d, d)) / np.sqrt(d),
                "wo": rng.standard_normal((d, d)) / np.sqrt(d),
                "w1": rng.standard_normal((d_ffn, d)) / np.sqrt(d),
                "w2": rng.standard_normal((d, d_ffn)) / np.sqrt(d_ffn),
            })
        self.head = rng.standard_normal((vocab, d)) / np.sqrt(d) * 4.0

    def forward(self, tokens):
        """Returns logits [T, V] and hidden states [L+1, T, d] (index l is the
        output of layer l; index 0 the embedding)."""
        x = self.embed[np.asarray(tokens)]
        T = x.shape[0]
        hs = [x]
        causal = np.triu(np.full((T, T), -np.inf), k=1)
        ones = np.ones(self.d)
        for p in self.layers:
            a = ref.rms_norm(x, ones, 1e-6)
            q = (a @ p["wq"].T).reshape(T, self.H, self.dh)
            k = (a @ p["wk"].T).reshape(T, self.H, self.dh)
            v = (a @ p["wv"].T).reshape(T, self.H, self.dh)
            o = np.zeros((T, self.H, self.dh))
            for h in range(self.H):
                s = q[:, h] @ k[:, h].T / np.sqrt(self.dh) + causal
                s = s - s.max(axis=-1, keepdims=True)
                w = np.exp(s)
                w /= w.sum(axis=-1, keepdims=True)
                o[:, h] = w @ v[:, h]
            x = x + o.reshape(T, self.d) @ p["wo"].T
            f = ref.rms_norm(x, ones, 1e-6)
            x = x + np.tanh(f @ p["w1"].T) @ p["w2"].T
            hs.append(x)
        logits = ref.rms_norm(x, ones, 1e-6) @ self.head.T
        return logits, np.stack(hs)

    def taps(self, hidden, rows):
        """[len(rows), n_taps, d] tapped states of the given positions."""
        return np.stack([hidden[l][rows] for l in tap_layers(self.L)], axis=1)


def greedy_generate(target: TinyTarget, prompt, n_new: int) -> list[int]:
    """Target-only greedy decoding: the reference stream."""
    seq = list(prompt)
    out = []
    while len(out) < n_new:
        logits, _ = target.forward(seq)
        t = int(ref.argmax_lowest(logits[-1]))
        seq.append(t)
        out.append(t)
    return out


class OracleDrafter:
    """The oracle drafter with its injected-context KV state for one sequence."""

    def __init__(self, cfg: ref.Cfg, W: dict):
        self.cfg, self.W = cfg, W
        self.k = [np.zeros((cfg.n_kv_heads, 0, cfg.head_dim)) for _ in range(cfg.n_layers)]
        self.v = [np.zeros((cfg.n_kv_heads, 0, cfg.head_dim)) for _ in range(cfg.n_layers)]

    @property
    def n_ctx(self) -> int:
        return self.k[0].shape[1]

    def inject(self, taps):
        """Fuse taps [T, n_taps, Dt] and append their K/V to every layer."""
        if len(taps) == 0:
            return
        h_ctx = ref.ctx_fuse(self.cfg, self.W["w_c"], self.W["g_c"], taps)
        for i in range(self.cfg.n_layers):
            k, v = ref.ctx_kv(self.cfg, self.W["w_qkv"][i], h_ctx, self.n_ctx)
            self.k[i] = np.concatenate([self.k[i], k], axis=1)
            self.v[i] = np.concatenate([self.v[i], v], axis=1)

    def draft(self, anchor: int, _seq) -> np.ndarray:
        out = ref.draft_block(self.cfg, self.W, anchor, self.k, self.v, self.n_ctx)
        return out["draft"]


def speculative_generate(target: TinyTarget, drafter, prompt, n_new: int,
                         gamma: int, stats: list | None = None) -> list[int]:
    """DFlash-style greedy speculative decoding.

    drafter.inject(taps) receives the tapped states of newly verified
    positions; drafter.draft(anchor, seq) returns gamma tokens. The target's
    prefill yields the first token; each cycle verifies [anchor, drafts] in
    one target pass and commits tau tokens (accepted drafts plus the bonus)."""
    seq = list(prompt)                      # tokens whose features are injected
    logits, hidden = target.forward(seq)
    drafter.inject(target.taps(hidden, np.arange(len(seq))))
    anchor = int(ref.argmax_lowest(logits[-1]))
    out = [anchor]
    while len(out) < n_new:
        d = np.asarray(drafter.draft(anchor, seq), dtype=np.int64)
        assert d.shape == (gamma,)
        block = seq + [anchor] + [int(x) for x in d]
        logits, hidden = target.forward(block)
        n0 = len(seq)
        tau, committed, nxt = ref.verify_accept(logits[n0:n0 + gamma + 1], d)
        if stats is not None:
            stats.append(tau)
        accepted_rows = np.arange(n0, n0 + tau)  # anchor + accepted drafts
        drafter.inject(target.taps(hidden, accepted_rows))
        seq = seq + [anchor] + [int(x) for x in d[: tau - 1]]
        out.extend(int(x) for x in committed[:tau])
        anchor = nxt
    return out[:n_new]


def cycle_seed(seed: int, cycle: int) -> int:
    """Per-cycle generator state: a splitmix64 output of (seed, cycle), so
    that every cycle draws from its own counter space."""
    return int(ref.rng_u64(seed, 15, 0, 0, cycle))


def speculative_sample_generate(target: TinyTarget, draft_logits_fn, prompt, anchor: int,
                                n_new: int, gamma: int, T: float, seed: int,
                                stats: list | None = None) -> list[int]:
    """Speculative decoding at temperature T from a given anchor ([P1] temp-1
    results; [P2] lossless rejection-acceptance paragraph): each cycle the
    drafter's logits [gamma, V] give sampled drafts (ref.draft_sample), the
    target scores [anchor, drafts] in one pass, and ref.verify_sample commits
    tau tokens. draft_logits_fn(anchor, seq) may be any drafter: the
    committed stream follows the target's sampling distribution regardless.
    Returns the first n_new committed tokens after the anchor."""
    seq = list(prompt)
    out = []
    cycle = 0
    while len(out) < n_new:
        s = cycle_seed(seed, cycle)
        ql = ref.f64(draft_logits_fn(anchor, seq))
        d = ref.draft_sample(ql, T, s, 0)
        block = seq + [anchor] + [int(x) for x in d]
        logits, _ = target.forward(block)
        n0 = len(seq)
        tau, committed, nxt = ref.verify_sample(logits[n0:n0 + gamma + 1], ql, d, T, s, 0)
        if stats is not None:
            stats.append(tau)
        seq = seq + [anchor] + [int(x) for x in d[: tau - 1]]
        out.extend(int(x) for x in committed[:tau])
        anchor = nxt
        cycle += 1
    return out[:n_new]


def target_sampling_pair_probs(target: TinyTarget, prompt, anchor: int, T: float) -> np.ndarray:
    """Exact P(first two tokens after the anchor = (y1, y2)) under target-only
    sampling at temperature T: p(y1 | prompt, anchor) * p(y2 | ..., y1)."""
    base = list(prompt) + [anchor]
    logits, _ = target.forward(base)
    p1 = ref.softmax_t(logits[-1], T)
    P = np.zeros((target.V, target.V))
    for y1 in range(target.V):
        l2, _ = target.forward(base + [y1])
        P[y1] = p1[y1] * ref.softmax_t(l2[-1], T)
    return P
