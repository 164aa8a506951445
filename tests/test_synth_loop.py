"""The draft-verify loop's synthetic target (input generation shared by the
loop's GPU test and the bench): per row, the token it makes the unique
argmax agrees with the drafted token with probability 0.8, decided by a hash
of the drafted token itself, never at the bonus row; elsewhere it is a
different token. E[tau] = 1 + sum_{k=1..16} 0.8^k = 4.89."""
import numpy as np
import torch

import synth
from oracle import dflash_ref as ref

WL = synth.Workload("loop_small", n_layers=1, d_target=64, n_taps=5, d_model=128, n_q_heads=2,
                    n_kv_heads=1, head_dim=64, d_ffn=128, vocab=5003, gamma=16, dtype="f32", batch=4,
                    ctx=64, cycles=8, seed=77)


def test_target_argmax_is_the_intended_token_and_unique():
    rng = np.random.default_rng(1)
    for cyc in range(3):
        draft = torch.as_tensor(rng.integers(0, WL.vocab, (WL.batch, WL.gamma)), dtype=torch.int32)
        tl = synth.loop_target_logits(WL, cyc, draft)
        key16, offset = synth.loop_plan(WL, cyc)
        want = synth.loop_intended(WL, torch.as_tensor(key16), torch.as_tensor(offset), draft)
        top2 = tl.topk(2, dim=-1).values
        assert (top2[..., 0] - top2[..., 1] >= 1.0 - 1e-6).all()       # unique argmax
        assert torch.equal(tl.argmax(-1), want)
        # not agreeing means a different token; the bonus row never agrees
        agree = want[:, :-1] == draft.to(torch.int64)
        assert not (want[:, -1] == -1).any()
        assert ((want[:, :-1] != draft.to(torch.int64)) == ~agree).all()


def test_agreement_rate_and_mean_acceptance():
    rng = np.random.default_rng(2)
    agree_n, taus = 0, []
    wl = WL.replace(batch=64)
    for cyc in range(40):
        draft = rng.integers(0, wl.vocab, (wl.batch, wl.gamma)).astype(np.int32)
        key16, offset = synth.loop_plan(wl, cyc)
        want = synth.loop_intended(wl, torch.as_tensor(key16), torch.as_tensor(offset),
                                   torch.as_tensor(draft)).numpy()
        agree_n += int((want[:, :-1] == draft).sum())
        for b in range(wl.batch):
            # tau = 1 + the length of the agreeing prefix
            t = 1
            for j in range(wl.gamma):
                if want[b, j] != draft[b, j]:
                    break
                t += 1
            taus.append(t)
    p = agree_n / (40 * wl.batch * wl.gamma)
    assert abs(p - 0.8) < 0.02, p
    assert abs(np.mean(taus) - (1 + sum(0.8 ** k for k in range(1, 17)))) < 0.35, np.mean(taus)


def test_agreement_depends_on_the_drafted_token():
    key16, offset = synth.loop_plan(WL, 0)
    k = torch.as_tensor(key16)
    o = torch.as_tensor(offset)
    outcomes = set()
    for tok in range(200):
        d = torch.full((WL.batch, WL.gamma), tok, dtype=torch.int32)
        outcomes.add(bool((synth.loop_intended(WL, k, o, d)[0, 0] == tok).item()))
    assert outcomes == {True, False}


def test_oracle_verify_on_synthetic_target_gives_tau_from_the_agreement_prefix():
    rng = np.random.default_rng(3)
    draft = torch.as_tensor(rng.integers(0, WL.vocab, (WL.batch, WL.gamma)), dtype=torch.int32)
    tl = synth.loop_target_logits(WL, 5, draft)
    key16, offset = synth.loop_plan(WL, 5)
    want = synth.loop_intended(WL, torch.as_tensor(key16), torch.as_tensor(offset), draft).numpy()
    for b in range(WL.batch):
        t, c, n = ref.verify_accept(tl[b].numpy(), draft[b].numpy())
        a = 0
        while a < WL.gamma and want[b, a] == int(draft[b, a]):
            a += 1
        assert t == a + 1 and n == want[b, a]
