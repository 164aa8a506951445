"""Pins of the CPU oracle against facts fixed by the pages and by mathematics
(closed forms, invariants, library routines, brute force on tiny inputs).
CPU only."""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import dflash_ref as ref
from oracle import spec_loop


def tiny_cfg(**kw):
    base = dict(n_layers=2, d_target=16, n_taps=5, d_model=32, n_q_heads=4,
                n_kv_heads=2, head_dim=8, d_ffn=48, vocab=40, gamma=4,
                mask_token_id=39, rms_eps=1e-6, rope_theta=1e4)
    base.update(kw)
    return ref.Cfg(**base)


def tiny_weights(cfg, seed=0):
    rng = np.random.default_rng(seed)
    L, D, Dt = cfg.n_layers, cfg.d_model, cfg.d_target
    Hq, Hkv, Dh, F_, V = (cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                          cfg.d_ffn, cfg.vocab)
    nqkv = (Hq + 2 * Hkv) * Dh

    def lin(*shape):
        return rng.standard_normal(shape) / np.sqrt(shape[-1])

    return {
        "w_c": lin(D, cfg.n_taps * Dt), "g_c": 1 + 0.1 * rng.standard_normal(D),
        "embed": rng.standard_normal((V, D)),
        "g_final": 1 + 0.1 * rng.standard_normal(D), "lm_head": lin(V, D),
        "g_attn": 1 + 0.1 * rng.standard_normal((L, D)), "w_qkv": lin(L, nqkv, D),
        "w_o": lin(L, D, Hq * Dh), "g_ffn": 1 + 0.1 * rng.standard_normal((L, D)),
        "w_gateup": lin(L, 2 * F_, D), "w_down": lin(L, D, F_),
    }


# ---------------------------------------------------------------- RMSNorm / fuse

def test_rmsnorm_unit_rms_with_unit_gain():
    x = np.random.default_rng(1).standard_normal((7, 64)) * 3.0
    y = ref.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-12)


@pytest.mark.parametrize("k", range(5))
def test_ctx_fuse_selects_tap_in_concat_order(k):
    """W_c = [0 .. I .. 0] (identity in block k) reduces H_t to RMSNorm of tap
    k: pins the feature-axis concatenation order l1..l5 and W_c's layout."""
    cfg = tiny_cfg(d_target=32, d_model=32)
    rng = np.random.default_rng(2)
    taps = rng.standard_normal((6, 5, 32))
    w_c = np.zeros((32, 5 * 32))
    w_c[:, k * 32:(k + 1) * 32] = np.eye(32)
    h = ref.ctx_fuse(cfg, w_c, np.ones(32), taps)
    x = taps[:, k, :]
    expect = x / (np.linalg.norm(x, axis=-1, keepdims=True) / np.sqrt(32))
    np.testing.assert_allclose(h, expect, rtol=1e-6)


def test_ctx_fuse_matches_torch_linear_rmsnorm():
    """[P4] §3.1 writes the fusion as nn.Linear (no bias) then nn.RMSNorm."""
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    taps = np.random.default_rng(3).standard_normal((9, 5 * cfg.d_target))
    got = ref.ctx_fuse(cfg, W["w_c"], W["g_c"], taps)
    t = torch.from_numpy(taps)
    u = F.linear(t, torch.from_numpy(W["w_c"]))
    want = F.rms_norm(u, (cfg.d_model,), torch.from_numpy(W["g_c"]), eps=cfg.rms_eps)
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- RoPE

def test_rope_is_complex_rotation():
    """Pair (j, j+Dh/2) as z = x_j + i x_{j+Dh/2}; RoPE multiplies z by
    exp(i * pos * theta^(-2j/Dh))."""
    rng = np.random.default_rng(4)
    dh, theta = 8, 100.0
    x = rng.standard_normal((5, 3, dh))
    pos = np.array([0, 1, 7, 300, 12345])
    y = ref.rope(x, pos, theta)
    for t in range(5):
        for h in range(3):
            for j in range(dh // 2):
                z = complex(x[t, h, j], x[t, h, j + dh // 2])
                w = z * complex(math.cos(pos[t] * theta ** (-2 * j / dh)),
                                math.sin(pos[t] * theta ** (-2 * j / dh)))
                assert abs(y[t, h, j] - w.real) < 1e-9
                assert abs(y[t, h, j + dh // 2] - w.imag) < 1e-9


def test_rope_relative_position_and_off_switch():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 1, 16))
    k = rng.standard_normal((1, 1, 16))

    def dot(m, n):
        return float(np.sum(ref.rope(q, np.array([m]), 1e4) * ref.rope(k, np.array([n]), 1e4)))

    assert abs(dot(3, 10) - dot(103, 110)) < 1e-9
    assert abs(dot(3, 10) - dot(10, 3)) > 1e-6   # not symmetric in general
    np.testing.assert_array_equal(ref.rope(q, np.array([5]), 0.0), q)
    np.testing.assert_allclose(np.linalg.norm(ref.rope(q, np.array([77]), 1e6)),
                               np.linalg.norm(q), rtol=1e-12)


# ---------------------------------------------------------------- attention

def brute_attention(cfg, q, k, v):
    """Pure-Python loops with math.exp: the textbook definition."""
    R, Hq, Dh = q.shape
    grp = cfg.n_q_heads // cfg.n_kv_heads
    out = np.zeros_like(q)
    for i in range(R):
        for h in range(Hq):
            g = h // grp
            n = k.shape[1]
            s = [sum(q[i, h, d] * k[g, j, d] for d in range(Dh)) / math.sqrt(Dh)
                 for j in range(n)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = sum(e)
            for d in range(Dh):
                out[i, h, d] = sum(e[j] * v[g, j, d] for j in range(n)) / z
    return out


@pytest.mark.parametrize("n", [0, 1, 5, 8])
def test_attention_brute_force_gqa(n):
    cfg = tiny_cfg(n_q_heads=4, n_kv_heads=2, head_dim=6)
    rng = np.random.default_rng(10 + n)
    q = rng.standard_normal((3, 4, 6))
    k = rng.standard_normal((2, n + 3, 6)) * 2
    v = rng.standard_normal((2, n + 3, 6))
    np.testing.assert_allclose(ref.attention(cfg, q, k, v),
                               brute_attention(cfg, q, k, v), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("n", [0, 37])
def test_attention_matches_torch_sdpa(n):
    """n = 0 is plain bidirectional attention inside the block; n > 0 is SDPA
    over the sequence-axis concatenation [ctx ; block] ([P4] §3.2)."""
    cfg = tiny_cfg(n_q_heads=8, n_kv_heads=2, head_dim=16)
    rng = np.random.default_rng(20 + n)
    R = 17
    q = rng.standard_normal((R, 8, 16))
    k = rng.standard_normal((2, n + R, 16))
    v = rng.standard_normal((2, n + R, 16))
    got = ref.attention(cfg, q, k, v)
    tq = torch.from_numpy(q).transpose(0, 1)                    # [H, R, Dh]
    tk = torch.from_numpy(k).repeat_interleave(4, dim=0)        # [H, n+R, Dh]
    tv = torch.from_numpy(v).repeat_interleave(4, dim=0)
    want = F.scaled_dot_product_attention(tq, tk, tv).transpose(0, 1)
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-10, atol=1e-12)


def test_attention_softmax_rows_sum_to_one():
    cfg = tiny_cfg()
    rng = np.random.default_rng(30)
    q = rng.standard_normal((5, 4, 8)) * 4
    k = rng.standard_normal((2, 40, 8)) * 4
    v = np.ones((2, 40, 8))
    np.testing.assert_allclose(ref.attention(cfg, q, k, v), 1.0, atol=1e-12)


def test_attention_dominant_key_returns_its_value():
    cfg = tiny_cfg(n_q_heads=2, n_kv_heads=1, head_dim=8)
    rng = np.random.default_rng(31)
    c = rng.standard_normal(8)
    q = c + 0.1 * rng.standard_normal((2, 2, 8))
    k = rng.standard_normal((1, 20, 8)) * 0.1
    v = rng.standard_normal((1, 20, 8))
    k[0, 13] = 1e3 * c
    out = ref.attention(cfg, q, k, v)
    for i in range(2):
        for h in range(2):
            np.testing.assert_allclose(out[i, h], v[0, 13], atol=1e-9)


def test_attention_gqa_equals_mha_with_repeated_kv():
    g = tiny_cfg(n_q_heads=6, n_kv_heads=2, head_dim=4)
    m = tiny_cfg(n_q_heads=6, n_kv_heads=6, head_dim=4)
    rng = np.random.default_rng(32)
    q = rng.standard_normal((3, 6, 4))
    k = rng.standard_normal((2, 9, 4))
    v = rng.standard_normal((2, 9, 4))
    np.testing.assert_allclose(ref.attention(g, q, k, v),
                               ref.attention(m, q, np.repeat(k, 3, 0), np.repeat(v, 3, 0)),
                               rtol=1e-12)


def test_attention_context_permutation_invariant():
    cfg = tiny_cfg()
    rng = np.random.default_rng(33)
    q = rng.standard_normal((4, 4, 8))
    k = rng.standard_normal((2, 30, 8))
    v = rng.standard_normal((2, 30, 8))
    perm = rng.permutation(30)
    np.testing.assert_allclose(ref.attention(cfg, q, k, v),
                               ref.attention(cfg, q, k[:, perm], v[:, perm]), rtol=1e-10)


# ---------------------------------------------------------------- KV injection

def test_ctx_kv_rows_are_wk_ht_and_append_invariant():
    cfg = tiny_cfg(rope_theta=0.0)
    W = tiny_weights(cfg)
    h = np.random.default_rng(40).standard_normal((11, cfg.d_model))
    k, v = ref.ctx_kv(cfg, W["w_qkv"][1], h, 0)
    nq = cfg.n_q_heads * cfg.head_dim
    nk = cfg.n_kv_heads * cfg.head_dim
    wk = W["w_qkv"][1][nq:nq + nk]
    wv = W["w_qkv"][1][nq + nk:]
    ek = np.einsum("td,nd->tn", h, wk).reshape(11, cfg.n_kv_heads, cfg.head_dim)
    ev = np.einsum("td,nd->tn", h, wv).reshape(11, cfg.n_kv_heads, cfg.head_dim)
    np.testing.assert_allclose(k, ek.transpose(1, 0, 2), rtol=1e-12)
    np.testing.assert_allclose(v, ev.transpose(1, 0, 2), rtol=1e-12)
    # position-independent without RoPE
    k5, _ = ref.ctx_kv(cfg, W["w_qkv"][1], h, 500)
    np.testing.assert_array_equal(k, k5)
    # with RoPE, injecting in two chunks equals one chunk
    cfg2 = tiny_cfg(rope_theta=1e4)
    ka, va = ref.ctx_kv(cfg2, W["w_qkv"][0], h, 3)
    k1, v1 = ref.ctx_kv(cfg2, W["w_qkv"][0], h[:4], 3)
    k2, v2 = ref.ctx_kv(cfg2, W["w_qkv"][0], h[4:], 7)
    np.testing.assert_allclose(ka, np.concatenate([k1, k2], 1), rtol=1e-12)
    np.testing.assert_allclose(va, np.concatenate([v1, v2], 1), rtol=1e-12)


# ---------------------------------------------------------------- drafter forward

def torch_draft_block_no_rope(cfg, W, anchor, k_ctx, v_ctx, n_ctx):
    """The drafter with RoPE off written with torch library layers
    (embedding, rms_norm, linear, scaled_dot_product_attention, silu)."""
    t = {k: torch.as_tensor(np.asarray(v, dtype=np.float64)) for k, v in W.items()}
    R, Hq, Hkv, Dh, F_ = cfg.rows, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_ffn
    nq, nk = Hq * Dh, Hkv * Dh
    ids = torch.tensor([anchor] + [cfg.mask_token_id] * cfg.gamma)
    h = F.embedding(ids, t["embed"])
    for i in range(cfg.n_layers):
        a = F.rms_norm(h, (cfg.d_model,), t["g_attn"][i], eps=cfg.rms_eps)
        qkv = F.linear(a, t["w_qkv"][i])
        q = qkv[:, :nq].reshape(R, Hq, Dh).transpose(0, 1)
        k = qkv[:, nq:nq + nk].reshape(R, Hkv, Dh).transpose(0, 1)
        v = qkv[:, nq + nk:].reshape(R, Hkv, Dh).transpose(0, 1)
        K = torch.cat([torch.as_tensor(k_ctx[i][:, :n_ctx]), k], 1)
        V = torch.cat([torch.as_tensor(v_ctx[i][:, :n_ctx]), v], 1)
        o = F.scaled_dot_product_attention(q, K, V, enable_gqa=True)
        h = h + F.linear(o.transpose(0, 1).reshape(R, nq), t["w_o"][i])
        f = F.rms_norm(h, (cfg.d_model,), t["g_ffn"][i], eps=cfg.rms_eps)
        gu = F.linear(f, t["w_gateup"][i])
        h = h + F.linear(F.silu(gu[:, :F_]) * gu[:, F_:], t["w_down"][i])
    z = F.rms_norm(h[1:], (cfg.d_model,), t["g_final"], eps=cfg.rms_eps)
    return F.linear(z, t["lm_head"]).numpy()


@pytest.mark.parametrize("n_ctx", [0, 13])
def test_draft_block_without_rope_matches_torch_layers(n_ctx):
    cfg = tiny_cfg(rope_theta=0.0)
    W = tiny_weights(cfg, seed=50)
    rng = np.random.default_rng(51)
    k_ctx = [rng.standard_normal((cfg.n_kv_heads, n_ctx, cfg.head_dim)) for _ in range(cfg.n_layers)]
    v_ctx = [rng.standard_normal((cfg.n_kv_heads, n_ctx, cfg.head_dim)) for _ in range(cfg.n_layers)]
    out = ref.draft_block(cfg, W, 7, k_ctx, v_ctx, n_ctx)
    want = torch_draft_block_no_rope(cfg, W, 7, k_ctx, v_ctx, n_ctx)
    np.testing.assert_allclose(out["logits"], want, rtol=1e-9, atol=1e-10)
    assert out["logits"].shape == (cfg.gamma, cfg.vocab)
    np.testing.assert_array_equal(out["draft"], want.argmax(-1))


def test_draft_block_with_zero_blocks_is_head_of_embedding():
    """With W_o = 0 and W_down = 0 every layer adds nothing, so the logits
    of each mask row are W_lm RMSNorm(E[mask]; g_final) (residual wiring and
    the final norm; only mask rows reach the head)."""
    cfg = tiny_cfg()
    W = tiny_weights(cfg, seed=52)
    W["w_o"] = np.zeros_like(W["w_o"])
    W["w_down"] = np.zeros_like(W["w_down"])
    k_ctx = [np.zeros((cfg.n_kv_heads, 0, cfg.head_dim))] * cfg.n_layers
    out = ref.draft_block(cfg, W, 3, k_ctx, k_ctx, 0, want_dumps=True)
    e = W["embed"][cfg.mask_token_id]
    z = W["g_final"] * e / np.sqrt(np.mean(e * e) + cfg.rms_eps)
    np.testing.assert_allclose(out["logits"], np.tile(W["lm_head"] @ z, (cfg.gamma, 1)), rtol=1e-12)
    for layer in range(cfg.n_layers + 1):
        np.testing.assert_array_equal(out["dumps"][layer][0], W["embed"][3])


def test_draft_rows_differ_by_position_with_rope():
    """Reading: without a positional code all mask rows would be equal."""
    cfg = tiny_cfg()
    W = tiny_weights(cfg, seed=53)
    k_ctx = [np.zeros((cfg.n_kv_heads, 0, cfg.head_dim))] * cfg.n_layers
    on = ref.draft_block(cfg, W, 3, k_ctx, k_ctx, 0)["logits"]
    off = ref.draft_block(ref.Cfg(**{**cfg.__dict__, "rope_theta": 0.0}), W, 3, k_ctx, k_ctx, 0)["logits"]
    assert np.abs(on[0] - on[1]).max() > 1e-3
    np.testing.assert_allclose(off[0], off[1], rtol=1e-12)


def test_argmax_ties_take_lowest_index():
    x = np.array([[0.0, 2.0, 2.0, 1.0], [5.0, 5.0, 5.0, 5.0]])
    np.testing.assert_array_equal(ref.argmax_lowest(x), [1, 0])


# ---------------------------------------------------------------- verify-accept

def onehot_logits(tokens, V):
    x = np.zeros((len(tokens), V))
    x[np.arange(len(tokens)), tokens] = 1.0
    return x


@pytest.mark.parametrize("gamma", [1, 2, 3, 4])
def test_verify_accept_brute_force(gamma):
    """Every draft in 3^gamma against every target sequence in 3^(gamma+1):
    tau - 1 is the largest k whose prefixes of length k agree."""
    for d in itertools.product(range(3), repeat=gamma):
        for t in itertools.product(range(3), repeat=gamma + 1):
            tau, committed, nxt = ref.verify_accept(onehot_logits(t, 3), np.array(d))
            k = max(k for k in range(gamma + 1) if list(d[:k]) == list(t[:k]))
            assert tau == k + 1 and 1 <= tau <= gamma + 1
            assert list(committed[:tau]) == list(d[:k]) + [t[k]]
            assert all(c == -1 for c in committed[tau:])
            assert nxt == t[k]


def test_verify_accept_extremes():
    V, g = 50, 16
    rng = np.random.default_rng(60)
    d = rng.integers(0, V, size=g)
    t = np.concatenate([d, [7]])
    tau, c, nxt = ref.verify_accept(onehot_logits(t, V), d)
    assert tau == g + 1 and list(c) == list(t) and nxt == 7
    t2 = t.copy()
    t2[0] = (d[0] + 1) % V
    tau, c, nxt = ref.verify_accept(onehot_logits(t2, V), d)
    assert tau == 1 and c[0] == t2[0] and nxt == t2[0] and all(c[1:] == -1)


# ---------------------------------------------------------------- lossless loop

def test_tap_layers_rule():
    """Five layers spread evenly from the second to the third-from-last."""
    assert spec_loop.tap_layers(8) == [2, 3, 4, 5, 6]
    assert spec_loop.tap_layers(36) == [2, 10, 18, 26, 34]


class TruthDrafter:
    """Proposes the target's own greedy continuation, corrupted at a seeded
    position with probability 0.7, so tau spreads over [1, gamma + 1]."""

    def __init__(self, target, gamma, seed):
        self.target, self.gamma = target, gamma
        self.rng = np.random.default_rng(seed)

    def inject(self, taps):
        pass

    def draft(self, anchor, seq):
        s = list(seq) + [anchor]
        out = []
        for _ in range(self.gamma):
            logits, _ = self.target.forward(s)
            t = int(np.argmax(logits[-1]))
            out.append(t)
            s.append(t)
        out = np.array(out)
        if self.rng.random() < 0.7:
            j = self.rng.integers(0, self.gamma)
            out[j] = (out[j] + 1 + self.rng.integers(0, self.target.V - 1)) % self.target.V
        return out


@pytest.mark.parametrize("drafter_kind", ["oracle", "truth"])
def test_speculative_decoding_is_lossless(drafter_kind):
    target = spec_loop.TinyTarget(seed=70)
    prompt = [1, 5, 9, 2, 33, 17]
    n_new, gamma = 40, 4
    want = spec_loop.greedy_generate(target, prompt, n_new)
    if drafter_kind == "oracle":
        cfg = tiny_cfg(d_target=target.d, vocab=target.V, mask_token_id=target.V - 1,
                       gamma=gamma)
        drafter = spec_loop.OracleDrafter(cfg, tiny_weights(cfg, seed=71))
    else:
        drafter = TruthDrafter(target, gamma, seed=72)
    stats = []
    got = spec_loop.speculative_generate(target, drafter, prompt, n_new, gamma, stats)
    assert got == want
    assert all(1 <= s <= gamma + 1 for s in stats)
    if drafter_kind == "truth":
        assert min(stats) == 1 and max(stats) == gamma + 1


def brute_draft_logits_1layer(cfg, W, anchor, h_ctx):
    """A one-layer drafter written with scalar loops and complex-number RoPE.
    Context row t sits at position t; block row i at position n + i, so the
    block continues the injected context (reading of the positional code)."""
    n, R, D = len(h_ctx), cfg.rows, cfg.d_model
    Hq, Hkv, Dh, F_ = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.d_ffn
    half = Dh // 2

    def rot(vec, p):
        out = list(vec)
        for j in range(half):
            w = cfg.rope_theta ** (-2.0 * j / Dh)
            z = complex(vec[j], vec[j + half]) * complex(math.cos(p * w), math.sin(p * w))
            out[j], out[j + half] = z.real, z.imag
        return out

    def norm(x, g):
        r = math.sqrt(sum(a * a for a in x) / len(x) + cfg.rms_eps)
        return [g[i] * x[i] / r for i in range(len(x))]

    def mv(w, x):
        return [sum(w[o][i] * x[i] for i in range(len(x))) for o in range(len(w))]

    wqkv = W["w_qkv"][0]
    nq, nk = Hq * Dh, Hkv * Dh
    keys = [[None] * (n + R) for _ in range(Hkv)]
    vals = [[None] * (n + R) for _ in range(Hkv)]
    for t in range(n):
        kk, vv = mv(wqkv[nq:nq + nk], h_ctx[t]), mv(wqkv[nq + nk:], h_ctx[t])
        for g in range(Hkv):
            keys[g][t] = rot(kk[g * Dh:(g + 1) * Dh], t)
            vals[g][t] = vv[g * Dh:(g + 1) * Dh]
    ids = [anchor] + [cfg.mask_token_id] * cfg.gamma
    h = [list(W["embed"][i]) for i in ids]
    a = [norm(h[i], W["g_attn"][0]) for i in range(R)]
    qs = []
    for i in range(R):
        qkv = mv(wqkv, a[i])
        qs.append([rot(qkv[hh * Dh:(hh + 1) * Dh], n + i) for hh in range(Hq)])
        for g in range(Hkv):
            keys[g][n + i] = rot(qkv[nq + g * Dh:nq + (g + 1) * Dh], n + i)
            vals[g][n + i] = qkv[nq + nk + g * Dh:nq + nk + (g + 1) * Dh]
    for i in range(R):
        o = []
        for hh in range(Hq):
            g = hh // (Hq // Hkv)
            s = [sum(qs[i][hh][d] * keys[g][j][d] for d in range(Dh)) / math.sqrt(Dh)
                 for j in range(n + R)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            o += [sum(e[j] * vals[g][j][d] for j in range(n + R)) / sum(e) for d in range(Dh)]
        h[i] = [h[i][c] + y for c, y in enumerate(mv(W["w_o"][0], o))]
    for i in range(R):
        f = norm(h[i], W["g_ffn"][0])
        gu = mv(W["w_gateup"][0], f)
        act = [gu[c] / (1 + math.exp(-gu[c])) * gu[F_ + c] for c in range(F_)]
        h[i] = [h[i][c] + y for c, y in enumerate(mv(W["w_down"][0], act))]
    return np.array([mv(W["lm_head"], norm(h[i], W["g_final"])) for i in range(1, R)])


def test_draft_block_one_layer_brute_force_with_rope():
    cfg = tiny_cfg(n_layers=1, d_model=16, n_q_heads=2, n_kv_heads=1, head_dim=4,
                   d_ffn=8, vocab=12, mask_token_id=11, gamma=3, rope_theta=10.0)
    W = tiny_weights(cfg, seed=54)
    h_ctx = np.random.default_rng(55).standard_normal((5, cfg.d_model))
    k, v = ref.ctx_kv(cfg, W["w_qkv"][0], h_ctx, 0)
    got = ref.draft_block(cfg, W, 4, [k], [v], 5)["logits"]
    want = brute_draft_logits_1layer(cfg, W, 4, h_ctx)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-11)
