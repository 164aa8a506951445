"""CPU oracle of the DFlash drafting step -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct numpy in float64. Only the test-suite, the
smoke check and the benchmark's CPU-baseline leg may import this module; the
product path never does. It shares no code with the CUDA library.

Each function states the passage it follows:
  [P1] "DFlash: Block Diffusion for Flash Speculative Decoding 논문 정리"
  [P2] "DFlash 블록 확산 디코딩: 투기적 디코딩의 드래프트 비용을 상수로 만드는 법"
  [P4] "ICML'26 | DFlash：用 Diffusion 模型干掉 AR Drafter，投机解码提速 6×"
Readings where the pages are silent (positional encoding, layer wiring,
epsilon, tie-breaking) are listed in the design notes and repeated here at
the point of use.

Library primitives used as single steps: matrix product (numpy @), exp,
sqrt, cos/sin, argmax. No blocking, fusion or reordering beyond the
definitions.
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class Cfg:
    n_layers: int
    d_target: int
    n_taps: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    gamma: int
    mask_token_id: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def rows(self) -> int:
        return self.gamma + 1


def f64(x) -> np.ndarray:
    """Any array-like (numpy, or a CPU torch tensor via numpy()) as float64."""
    if hasattr(x, "detach"):
        x = x.detach().float().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


# -- building blocks ---------------------------------------------------------

def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: g * x / sqrt(mean(x^2) + eps).
    [P1] "KV Injection 메커니즘" (H_t = RMSNorm(...)); [P4] §3.1 (nn.RMSNorm)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return g * x / np.sqrt(ms + eps)


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """x @ w^T for a row-major [out, in] weight (a linear layer without bias)."""
    return x @ f64(w).T


def rope(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotary position encoding of x [..., T, H, Dh] at positions pos [T].

    The pages name no positional encoding; without one the gamma mask rows
    are identical inputs and would draft identical tokens. Reading: the
    rotate-half form used by the Qwen3 family. Dimension j and j + Dh/2 are
    rotated together by the angle pos * theta^(-2j/Dh). theta == 0 disables
    it (the literal formulas of [P1] "KV Injection 메커니즘")."""
    if theta == 0:
        return x
    dh = x.shape[-1]
    half = dh // 2
    j = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * j / dh)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]  # [T, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def argmax_lowest(x: np.ndarray) -> np.ndarray:
    """argmax over the last axis; numpy returns the first (lowest) index of
    the maximum, the tie rule of torch.argmax used in [P4] §3.3."""
    assert np.all(np.isfinite(x)), "oracle assumes finite logits"
    return np.argmax(x, axis=-1)


# -- a1: context fusion ------------------------------------------------------

def ctx_fuse(cfg: Cfg, w_c, g_c, taps) -> np.ndarray:
    """H_t = RMSNorm(W_c [H(l1); ...; H(l5)]), [P1] "KV Injection 메커니즘"
    and [P4] §3.1: the tapped states of one token are concatenated on the
    feature axis in tap order, projected by W_c [D, 5*Dt], then RMS-normed.
    taps: [T, n_taps, Dt] or [T, n_taps*Dt]. Returns [T, D]."""
    x = f64(taps)
    x = x.reshape(x.shape[0], cfg.n_taps * cfg.d_target)
    u = linear(x, w_c)
    return rms_norm(u, f64(g_c), cfg.rms_eps)


# -- a2: KV injection ----------------------------------------------------------

def split_qkv(cfg: Cfg, w_qkv_layer):
    """Row blocks of one layer's stacked projection: W^Q, W^K, W^V."""
    w = f64(w_qkv_layer)
    nq = cfg.n_q_heads * cfg.head_dim
    nk = cfg.n_kv_heads * cfg.head_dim
    return w[:nq], w[nq:nq + nk], w[nq + nk:nq + 2 * nk]


def ctx_kv(cfg: Cfg, w_qkv_layer, h_ctx, pos0: int, positions=None):
    """Injected context entries of one layer, [P1] "KV Injection 메커니즘":
    the first (context) part of K_i = [W_i^K H_t ; W_i^K H_d]_seq and of V_i.
    Row t sits at absolute position pos0 + t (or positions[t] when given);
    RoPE applies to K (reading). Returns K, V as [Hkv, T, Dh]."""
    _, wk, wv = split_qkv(cfg, w_qkv_layer)
    h = f64(h_ctx)
    T = h.shape[0]
    k = linear(h, wk).reshape(T, cfg.n_kv_heads, cfg.head_dim)
    v = linear(h, wv).reshape(T, cfg.n_kv_heads, cfg.head_dim)
    pos = pos0 + np.arange(T) if positions is None else np.asarray(positions)
    k = rope(k, pos, cfg.rope_theta)
    return k.transpose(1, 0, 2), v.transpose(1, 0, 2)


# -- a5: attention -------------------------------------------------------------

def attention(cfg: Cfg, q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """softmax(q K^T / sqrt(Dh)) V with grouped KV heads and no mask.

    [P4] §3.2 (scaled dot-product attention over the concatenated K, V;
    bidirectional inside the block); [P1] "추론 구조" (mask positions decoded
    with bidirectional attention). Query head h reads KV head
    h // (Hq / Hkv) (reading for GQA). Softmax subtracts the row max.
    q: [R, Hq, Dh]; k, v: [Hkv, n, Dh]. Returns [R, Hq, Dh]."""
    R = q.shape[0]
    grp = cfg.n_q_heads // cfg.n_kv_heads
    out = np.zeros((R, cfg.n_q_heads, cfg.head_dim))
    scale = 1.0 / np.sqrt(cfg.head_dim)
    for h in range(cfg.n_q_heads):
        g = h // grp
        s = (q[:, h, :] @ k[g].T) * scale          # [R, n]
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=-1, keepdims=True)
        out[:, h, :] = p @ v[g]
    return out


# -- a3..a8: one-pass block drafting ------------------------------------------

def draft_block(cfg: Cfg, W: dict, anchor: int, k_ctx, v_ctx, n_ctx: int,
                want_dumps: bool = False, ids=None) -> dict:
    """One drafting pass for one sequence, [P4] §3.3 and §3.2, [P1] "추론 구조":

      input ids  [anchor, m, ..., m] (R = gamma + 1 rows), positions
                 n_ctx + 0 .. n_ctx + gamma
      h          = Embed(ids)
      per layer i (pre-norm wiring with residuals -- reading):
        a        = RMSNorm(h; g_attn_i)
        q, k, v  = W_i^Q a, W_i^K a, W_i^V a ; RoPE on q and k
        K_i, V_i = [K_ctx_i ; k], [V_ctx_i ; v]   (sequence-axis concatenation)
        h       += W_i^O attention(q, K_i, V_i)
        f        = RMSNorm(h; g_ffn_i)
        h       += W_i^down(silu(W_i^gate f) * W_i^up f)
      z      = RMSNorm(h[1:]; g_final)   (only the mask rows reach the head)
      logits = W_lm z ; draft = argmax (lowest index on ties)

    W: stacked weights (arrays or CPU tensors, any float dtype).
    k_ctx, v_ctx: per layer [Hkv, >= n_ctx, Dh] injected entries.
    ids: optional block input [R] (row 0 the anchor) replacing [anchor, m, ..., m]
    -- the partially unmasked block of multi-step drafting.
    Returns dict(logits [gamma, V], draft [gamma], dumps [L+1, R, D] or None)."""
    L, R, D = cfg.n_layers, cfg.rows, cfg.d_model
    Hq, Hkv, Dh, F = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_ffn
    eps = cfg.rms_eps
    ids = np.array([anchor] + [cfg.mask_token_id] * cfg.gamma) if ids is None else np.asarray(ids)
    assert ids.shape == (R,) and ids[0] == anchor
    pos = n_ctx + np.arange(R)
    h = f64(W["embed"][ids])
    dumps = [h.copy()] if want_dumps else None
    for i in range(L):
        a = rms_norm(h, f64(W["g_attn"][i]), eps)
        wq, wk, wv = split_qkv(cfg, W["w_qkv"][i])
        q = rope((a @ wq.T).reshape(R, Hq, Dh), pos, cfg.rope_theta)
        k = rope((a @ wk.T).reshape(R, Hkv, Dh), pos, cfg.rope_theta)
        v = (a @ wv.T).reshape(R, Hkv, Dh)
        K = np.concatenate([f64(k_ctx[i])[:, :n_ctx], k.transpose(1, 0, 2)], axis=1)
        V = np.concatenate([f64(v_ctx[i])[:, :n_ctx], v.transpose(1, 0, 2)], axis=1)
        o = attention(cfg, q, K, V).reshape(R, Hq * Dh)
        h = h + linear(o, W["w_o"][i])
        f = rms_norm(h, f64(W["g_ffn"][i]), eps)
        wgu = f64(W["w_gateup"][i])
        gate = f @ wgu[:F].T
        up = f @ wgu[F:].T
        h = h + linear(silu(gate) * up, W["w_down"][i])
        if want_dumps:
            dumps.append(h.copy())
    z = rms_norm(h[1:], f64(W["g_final"]), eps)
    logits = linear(z, W["lm_head"])
    return {"logits": logits, "draft": argmax_lowest(logits),
            "dumps": np.stack(dumps) if want_dumps else None}


# -- a9: greedy verify-accept ----------------------------------------------------

def verify_accept(target_logits, draft):
    """Greedy verification, [P1] "Preliminaries" eq. (1) (tau counts the
    accepted drafts plus the target's bonus token, 1 <= tau <= gamma + 1) and
    "추론 구조" (the target checks the whole block in parallel).

    Row j of target_logits [gamma+1, V] is the target's next-token
    prediction after the anchor and draft[0..j-1]. Draft j is accepted while
    every earlier one was and it equals that prediction; the first
    prediction not matched (or the one after the last draft) is the bonus.
    Returns (tau, committed [gamma+1] padded with -1, next_anchor)."""
    t = argmax_lowest(f64(target_logits))
    d = np.asarray(draft)
    gamma = d.shape[0]
    a = 0
    while a < gamma and d[a] == t[a]:
        a += 1
    committed = np.full(gamma + 1, -1, dtype=np.int64)
    committed[:a] = d[:a]
    committed[a] = t[a]
    return a + 1, committed, int(t[a])


# -- NEXT: sampling (temperature > 0) draft and verification -------------------
#
# [P1] result tables "Qwen3-8B, temp 1" rows and [P2] "DFlash는 손실 없는 가속을
# 보장한다" paragraph: at temperature 1 the draft is sampled and verified by
# rejection-acceptance sampling, so the committed tokens follow the target's
# own sampling distribution. The pages name the mechanism but print no
# formula; the reading is standard speculative sampling:
#   q_j = softmax(drafter logits_j / T), x_j ~ q_j;
#   p_j = softmax(target logits_j / T);
#   draft j is accepted while r_j * q_j(x_j) < p_j(x_j), r_j ~ U(0, 1);
#   at the first rejection a the replacement is drawn from
#   norm(max(p_a - q_a, 0)); if all gamma are accepted the bonus is drawn
#   from p_gamma.
# Categorical draws use the Gumbel-max rule: argmax_v (log w_v + g_v) with
# g_v = -ln(-ln u_v) is a draw from w / sum(w).
#
# Random numbers: one counter-based generator, splitmix64 (Steele, Lea and
# Flood, "Fast splittable pseudorandom number generators", 2014; Vigna's
# reference splitmix64.c): the (c+1)-th output of the sequence started at
# state `seed` is mix(seed + (c + 1) * 0x9E3779B97F4A7C15 mod 2^64). The
# counter of a draw is c = stream * 2^60 + j * 2^52 + b * 2^32 + v, streams
# 0 draft sample, 1 residual sample, 2 bonus sample, 3 acceptance uniform.
# A uniform in (0, 1) is ((z >> 41) + 1/2) * 2^-23 (exact in float32).

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
STREAM_DRAFT, STREAM_RESID, STREAM_BONUS, STREAM_ACCEPT = 0, 1, 2, 3


def rng_u64(seed: int, stream: int, j: int, b: int, v) -> np.ndarray:
    """splitmix64 outputs for counters (stream, j, b, v); v an int or array."""
    with np.errstate(over="ignore"):
        c = (np.uint64(stream) << np.uint64(60)) | (np.uint64(j) << np.uint64(52)) | \
            (np.uint64(b) << np.uint64(32)) | np.asarray(v, dtype=np.uint64)
        z = np.uint64(seed) + (c + np.uint64(1)) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        return z ^ (z >> np.uint64(31))


def rng_uniform(seed: int, stream: int, j: int, b: int, v) -> np.ndarray:
    """Uniform in (0, 1) with 23 random bits: ((z >> 41) + 0.5) / 2^23, a
    value float32 holds exactly."""
    z = rng_u64(seed, stream, j, b, v)
    return ((z >> np.uint64(41)).astype(np.float64) + 0.5) / float(1 << 23)


def gumbel(seed: int, stream: int, j: int, b: int, n: int) -> np.ndarray:
    """Standard Gumbel noise -ln(-ln u) for v = 0 .. n-1."""
    u = rng_uniform(seed, stream, j, b, np.arange(n, dtype=np.uint64))
    return -np.log(-np.log(u))


def softmax_t(logits: np.ndarray, T: float) -> np.ndarray:
    """softmax(logits / T) over the last axis, by max subtraction."""
    z = f64(logits) / T
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def gumbel_argmax(score: np.ndarray, g: np.ndarray) -> int:
    """Categorical draw by the Gumbel-max rule over entries with finite score
    (score = log weight, -inf for weight 0); ties -> lowest index."""
    return int(np.argmax(score + g))


def draft_sample(logits, T: float, seed: int, b: int) -> np.ndarray:
    """Draft tokens x_j ~ softmax(logits_j / T) for mask rows j = 0..gamma-1
    of sequence b (stream 0)."""
    lg = f64(logits)
    V = lg.shape[-1]
    return np.array([gumbel_argmax(lg[j] / T, gumbel(seed, STREAM_DRAFT, j, b, V))
                     for j in range(lg.shape[0])], dtype=np.int64)


def accept_probability(p: np.ndarray, q: np.ndarray, x: int) -> float:
    """min(1, p(x) / q(x)): the chance that draft x, drawn from q, is kept."""
    return 1.0 if q[x] <= p[x] else p[x] / q[x]


def residual_distribution(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """norm(max(p - q, 0)); p itself when p == q everywhere (no residual mass)."""
    w = np.maximum(p - q, 0.0)
    s = w.sum()
    return w / s if s > 0 else p


def verify_sample(target_logits, draft_logits, draft, T: float, seed: int, b: int):
    """Rejection-acceptance verification of one block of sequence b.
    target_logits [gamma+1, V] (row j: target distribution after the anchor
    and draft[0..j-1]); draft_logits [gamma, V]; draft [gamma].
    Returns (tau, committed [gamma+1] padded with -1, next_anchor)."""
    p = softmax_t(target_logits, T)
    q = softmax_t(draft_logits, T)
    d = np.asarray(draft)
    gamma, V = d.shape[0], p.shape[-1]
    a = 0
    while a < gamma:
        r = float(rng_uniform(seed, STREAM_ACCEPT, a, b, 0))
        if r * q[a, d[a]] < p[a, d[a]]:
            a += 1
        else:
            break
    if a < gamma:
        w = residual_distribution(p[a], q[a])
        with np.errstate(divide="ignore"):
            y = gumbel_argmax(np.log(w), gumbel(seed, STREAM_RESID, a, b, V))
    else:
        y = gumbel_argmax(f64(target_logits)[gamma] / T, gumbel(seed, STREAM_BONUS, gamma, b, V))
    committed = np.full(gamma + 1, -1, dtype=np.int64)
    committed[:a] = d[:a]
    committed[a] = y
    return a + 1, committed, int(y)


# -- NEXT: multi-step confidence unmasking within a block --------------------
#
# [P2] "블록 확산 디코딩" drafting paragraph: the block starts as [MASK] at
# every position; each pass predicts all masked positions at once
# (bidirectional attention inside the block); the positions predicted with
# the highest confidence are unmasked first (their [MASK] replaced by the
# predicted token), and the passes repeat until the whole block is filled;
# the target then verifies the block at once. The pages give no schedule.
# Readings: confidence = max_v softmax(logits_j); S passes; pass s (0-based)
# unmasks ceil(m / (S - s)) of the m positions still masked; ties of
# confidence go to the lower position; an unmasked position keeps its token
# as input to later passes.


def confidence(logits) -> np.ndarray:
    """max_v softmax(logits_j): 1 / sum_v exp(l_v - max_v l)."""
    lg = f64(logits)
    return 1.0 / np.exp(lg - lg.max(axis=-1, keepdims=True)).sum(axis=-1)


def unmask_step(ids, logits, steps_left: int, mask_id: int):
    """One unmasking decision for one block. ids [R] (row 0 the anchor),
    logits [gamma, V] of the pass on ids. Returns the new ids [R]."""
    ids = np.array(ids, dtype=np.int64)
    masked = [j for j in range(ids.shape[0] - 1) if ids[j + 1] == mask_id]
    if not masked:
        return ids
    k = -(-len(masked) // steps_left)              # ceil(m / steps_left)
    conf = confidence(logits)
    order = sorted(masked, key=lambda j: (-conf[j], j))
    tok = argmax_lowest(f64(logits))
    for j in order[:k]:
        ids[j + 1] = tok[j]
    return ids


def draft_block_iterative(cfg: Cfg, W: dict, anchor: int, k_ctx, v_ctx, n_ctx: int,
                          n_steps: int) -> dict:
    """Multi-step drafting of one block: n_steps passes of draft_block, each
    followed by unmask_step. Returns dict(draft [gamma], ids per step
    [n_steps + 1, R], logits per step [n_steps, gamma, V])."""
    ids = np.array([anchor] + [cfg.mask_token_id] * cfg.gamma, dtype=np.int64)
    hist, lgs = [ids.copy()], []
    for s in range(n_steps):
        out = draft_block(cfg, W, anchor, k_ctx, v_ctx, n_ctx, ids=ids)
        lgs.append(out["logits"])
        ids = unmask_step(ids, out["logits"], n_steps - s, cfg.mask_token_id)
        hist.append(ids.copy())
    return {"draft": ids[1:], "ids": np.stack(hist), "logits": np.stack(lgs)}
