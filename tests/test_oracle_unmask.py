"""Pins of the oracle's multi-step confidence unmasking (a drafting variant
where the most confident masked positions are filled first, pass after pass)
against closed forms and the properties its reading fixes. CPU only."""
import numpy as np
import pytest

from oracle import dflash_ref as ref
from tests.test_oracle_pins import tiny_cfg, tiny_weights

scipy_special = pytest.importorskip("scipy.special")


def ctx_kv_random(cfg, n, seed):
    rng = np.random.default_rng(seed)
    k = [rng.standard_normal((cfg.n_kv_heads, n, cfg.head_dim)) for _ in range(cfg.n_layers)]
    v = [rng.standard_normal((cfg.n_kv_heads, n, cfg.head_dim)) for _ in range(cfg.n_layers)]
    return k, v


def test_confidence_is_the_largest_softmax_probability():
    lg = np.random.default_rng(1).standard_normal((5, 40)) * 3
    np.testing.assert_allclose(ref.confidence(lg), scipy_special.softmax(lg, axis=-1).max(axis=-1),
                               rtol=1e-13)
    assert ref.confidence(np.zeros((1, 8)))[0] == pytest.approx(1 / 8)
    assert ref.confidence(np.array([[0.0, 800.0, 0.0]]))[0] == pytest.approx(1.0)


@pytest.mark.parametrize("n_steps", [1, 2, 3, 5, 16])
def test_schedule_order_and_persistence_of_unmasked_tokens(n_steps):
    cfg = tiny_cfg(gamma=8)
    W = tiny_weights(cfg, seed=3)
    k, v = ctx_kv_random(cfg, 11, 4)
    out = ref.draft_block_iterative(cfg, W, 2, k, v, 11, n_steps)
    ids, lgs, m = out["ids"], out["logits"], cfg.mask_token_id
    masked = cfg.gamma
    for s in range(n_steps):
        before, after = ids[s], ids[s + 1]
        newly = [j for j in range(cfg.gamma) if before[j + 1] == m and after[j + 1] != m]
        still = [j for j in range(cfg.gamma) if after[j + 1] == m]
        # schedule: ceil(masked / steps left) positions per pass
        assert len(newly) == -(-masked // (n_steps - s))
        masked -= len(newly)
        assert len(still) == masked
        # tokens already placed never change
        keep = before[1:] != m
        np.testing.assert_array_equal(after[1:][keep], before[1:][keep])
        # the chosen positions take the pass's argmax and are at least as
        # confident as every position left masked
        conf = ref.confidence(lgs[s])
        tok = ref.argmax_lowest(lgs[s])
        for j in newly:
            assert after[j + 1] == tok[j]
            assert all(conf[j] >= conf[i] for i in still)
        # the pass saw the tokens placed so far
        np.testing.assert_array_equal(ref.draft_block(cfg, W, 2, k, v, 11, ids=before)["logits"], lgs[s])
    assert masked == 0 and (out["draft"] != m).all()


def test_one_pass_is_the_single_pass_draft():
    cfg = tiny_cfg(gamma=8)
    W = tiny_weights(cfg, seed=5)
    k, v = ctx_kv_random(cfg, 7, 6)
    one = ref.draft_block_iterative(cfg, W, 3, k, v, 7, 1)
    np.testing.assert_array_equal(one["draft"], ref.draft_block(cfg, W, 3, k, v, 7)["draft"])


def test_rows_that_see_only_themselves_unmask_in_position_order():
    # with W_o = W_down = 0 a row's logits depend on its own input token alone:
    # every masked row is identical, confidence ties, the lowest positions go
    # first, and every position takes the head of RMSNorm(E[m])'s argmax
    cfg = tiny_cfg(gamma=6)
    W = tiny_weights(cfg, seed=7)
    W["w_o"] = np.zeros_like(W["w_o"])
    W["w_down"] = np.zeros_like(W["w_down"])
    k, v = ctx_kv_random(cfg, 5, 8)
    out = ref.draft_block_iterative(cfg, W, 1, k, v, 5, 3)
    m = cfg.mask_token_id
    head = ref.argmax_lowest(ref.rms_norm(W["embed"][m], W["g_final"], cfg.rms_eps) @ W["lm_head"].T)
    assert (out["draft"] == head).all()
    # 6 masked, 3 passes: positions 0-1, then 2-3, then 4-5
    assert [list(np.nonzero(ids[1:] != m)[0]) for ids in out["ids"]] == [[], [0, 1], [0, 1, 2, 3],
                                                                          [0, 1, 2, 3, 4, 5]]


def test_more_passes_change_the_draft():
    # tokens placed early condition the later passes (bidirectional block)
    cfg = tiny_cfg(gamma=8)
    differs = 0
    for seed in range(6):
        W = tiny_weights(cfg, seed=seed)
        k, v = ctx_kv_random(cfg, 9, seed + 10)
        a = ref.draft_block_iterative(cfg, W, 4, k, v, 9, 1)["draft"]
        b = ref.draft_block_iterative(cfg, W, 4, k, v, 9, 4)["draft"]
        differs += int((a != b).any())
    assert differs > 0
