"""GPU parity of the sampling (temperature > 0) path: the sampled drafting pass
and the rejection-acceptance verifier against the oracle's definitions, and
the GPU verifier's committed tokens against the target distribution."""
import numpy as np
import pytest
import torch

import synth
from oracle import dflash_ref as ref
from tests import harness as H
from tests.test_gpu_parity import SMALL, run_chain

pytestmark = pytest.mark.gpu

DRAW_MARGIN = 1e-4     # score gap below which fp32 and fp64 Gumbel draws may part
ACCEPT_MARGIN = 1e-4   # relative gap |u q - p| / p below which an acceptance may flip


@pytest.fixture(scope="module")
def dfl(lib):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return lib


def oracle_draws(logits, T, seed, b):
    """Oracle Gumbel-max draws of each row with the top-2 score gap."""
    lg = ref.f64(logits)
    out, gaps = [], []
    for j in range(lg.shape[0]):
        s = lg[j] / T + ref.gumbel(seed, ref.STREAM_DRAFT, j, b, lg.shape[1])
        top = np.sort(s)[-2:]
        out.append(int(np.argmax(s)))
        gaps.append(top[1] - top[0])
    return np.array(out), np.array(gaps)


@pytest.mark.parametrize("T,seed", [(1.0, 11), (0.6, 2**63 + 5)])
def test_sampled_draft_is_the_gumbel_max_draw_of_the_logits(dfl, T, seed):
    gd = run_chain(dfl, SMALL, [300, 45, 0], check_dumps=False)
    wl = gd.wl
    B = wl.batch
    anchors = synth.anchors(wl)
    greedy, glogits, _ = gd.draft(anchors, 300, want_logits=True)
    a = torch.as_tensor(np.asarray(anchors, dtype=np.int32), device="cuda")
    draft = torch.empty((B, wl.gamma), dtype=torch.int32, device="cuda")
    logits = torch.empty((B, wl.gamma, wl.vocab), dtype=torch.float32, device="cuda")
    dfl.dflash_draft_block_sample(gd.cfg, gd.w, a, gd.ctx_len[:B], 300, gd.k_cache, gd.v_cache, T, seed,
                                  draft, logits, gd.status, gd.ws)
    torch.cuda.synchronize()
    gd.check_status()
    # the sampling pass computes the same logits as the greedy pass (checked
    # against the oracle by run_chain) ...
    assert torch.equal(logits, glogits)
    # ... and draws each token by Gumbel-max with the splitmix64 noise
    d = draft.cpu().numpy()
    n_tie = 0
    for b in range(B):
        want, gaps = oracle_draws(logits[b].cpu(), T, seed, b)
        bad = (d[b] != want) & (gaps >= DRAW_MARGIN)
        assert not bad.any(), (b, np.nonzero(bad), d[b], want)
        n_tie += int((d[b] != want).sum())
    H.report(f"sampled draft T={T}", "tokens_differing_at_draw_ties", n_tie, 0)
    # sampling is not greedy: some token differs from the argmax
    assert (d != greedy.cpu().numpy()).any()


def oracle_verify_with_margins(tl, dl, draft, T, seed, b):
    """ref.verify_sample plus the relative margins of its decisions."""
    tau, com, nxt = ref.verify_sample(tl, dl, draft, T, seed, b)
    p, q = ref.softmax_t(tl, T), ref.softmax_t(dl, T)
    a = tau - 1
    acc_margins = []
    for j in range(min(a + 1, len(draft))):
        u = float(ref.rng_uniform(seed, ref.STREAM_ACCEPT, j, b, 0))
        x = int(draft[j])
        acc_margins.append(abs(u * q[j, x] - p[j, x]) / max(p[j, x], u * q[j, x], 1e-300))
    V = p.shape[1]
    if a < len(draft):
        w = ref.residual_distribution(p[a], q[a])
        with np.errstate(divide="ignore"):
            s = np.log(w) + ref.gumbel(seed, ref.STREAM_RESID, a, b, V)
    else:
        s = ref.f64(tl)[a] / T + ref.gumbel(seed, ref.STREAM_BONUS, a, b, V)
    top = np.sort(s[np.isfinite(s)])[-2:]
    draw_margin = top[1] - top[0] if top.size == 2 else np.inf
    return tau, com, nxt, min(acc_margins) if acc_margins else np.inf, draw_margin


def planted_sampling_inputs(B, gamma, V, seed):
    g = torch.Generator().manual_seed(seed)
    tl = torch.randn((B, gamma + 1, V), generator=g) * 2.0
    dl = torch.randn((B, gamma, V), generator=g) * 2.0
    for b in range(B):
        if b % 2 == 0:       # a drafter close to the target: long accepted prefixes
            dl[b] = tl[b, :gamma] + 0.05 * torch.randn((gamma, V), generator=g)
    return tl, dl


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,V,T", [(2, 151936, 1.0), (5, 1003, 0.7), (3, 4103, 1.3)])
def test_verify_sample_matches_the_oracle(dfl, dtype, B, V, T):
    wl = SMALL.replace(batch=B, vocab=V)
    gd = H.GpuDrafter(dfl, wl, max_rows=16, weights=synth.weights(SMALL.replace(vocab=V), "cuda"))
    gamma, seed = wl.gamma, 1234 + V
    tl, dl = planted_sampling_inputs(B, gamma, V, seed)
    tl = tl.to(dtype)                                   # the verifier reads these values
    draft = np.stack([ref.draft_sample(dl[b], T, seed, b) for b in range(B)]).astype(np.int32)
    tau = torch.empty(B, dtype=torch.int32, device="cuda")
    committed = torch.empty((B, gamma + 1), dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    dfl.dflash_verify_sample(gd.cfg, tl.cuda(), dl.cuda(), torch.as_tensor(draft, device="cuda"), T, seed,
                             tau, committed, nxt, gd.ws)
    torch.cuda.synchronize()
    tau, committed, nxt = tau.cpu().numpy(), committed.cpu().numpy(), nxt.cpu().numpy()
    taus = []
    for b in range(B):
        t, c, n, acc_m, draw_m = oracle_verify_with_margins(tl[b].float(), dl[b], draft[b], T, seed, b)
        taus.append(t)
        if tau[b] != t:
            assert acc_m < ACCEPT_MARGIN, (b, tau[b], t, acc_m)
            continue
        if nxt[b] != n:
            assert draw_m < DRAW_MARGIN, (b, nxt[b], n, draw_m)
            continue
        np.testing.assert_array_equal(committed[b], c)
    H.report(f"verify_sample B={B} V={V} {dtype}", "oracle tau", float(np.mean(taus)), 0)
    assert max(taus) > 1          # the planted close drafters get drafts accepted


def test_verify_sample_commits_tokens_distributed_as_the_target(dfl):
    """Lossless in distribution on the GPU: with drafts drawn from q, the first
    committed token of every sequence is a draw from p_0."""
    V, gamma, T, B = 6, 3, 0.9, 64
    wl = SMALL.replace(batch=B, vocab=V, gamma=gamma)
    gd = H.GpuDrafter(dfl, wl, max_rows=16, weights=synth.weights(wl, "cuda"))
    g = torch.Generator().manual_seed(77)
    tl1 = torch.randn((gamma + 1, V), generator=g) * 1.5
    dl1 = torch.randn((gamma, V), generator=g) * 1.5
    tl = tl1.expand(B, gamma + 1, V).contiguous()
    dl = dl1.expand(B, gamma, V).contiguous()
    counts = np.zeros(V)
    tau = torch.empty(B, dtype=torch.int32, device="cuda")
    committed = torch.empty((B, gamma + 1), dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    mismatches = 0
    for call in range(50):
        seed = 9000 + call
        draft = np.stack([ref.draft_sample(dl1, T, seed, b) for b in range(B)]).astype(np.int32)
        dfl.dflash_verify_sample(gd.cfg, tl.cuda(), dl.cuda(), torch.as_tensor(draft, device="cuda"), T,
                                 seed, tau, committed, nxt, gd.ws)
        c = committed.cpu().numpy()
        for b in range(B):
            counts[c[b, 0]] += 1
            mismatches += int(c[b, 0] != ref.verify_sample(tl1, dl1, draft[b], T, seed, b)[1][0])
    from tests.test_oracle_sampling import chi2_pvalue
    assert chi2_pvalue(counts, ref.softmax_t(tl1[0], T)) > 1e-3
    assert mismatches == 0
