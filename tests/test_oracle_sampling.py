"""Pins of the oracle's sampling (temperature > 0) draft and verification
against facts fixed outside it: the published splitmix64 sequence, the
definition of its counter form, the Gumbel-max theorem, the speculative-
sampling identity (the committed token follows p exactly), and Monte Carlo
frequencies of the implemented procedure. CPU only."""
import numpy as np
import pytest

from oracle import dflash_ref as ref
from oracle import spec_loop as sl

scipy_stats = pytest.importorskip("scipy.stats")

M64 = (1 << 64) - 1
PHI = 0x9E3779B97F4A7C15


def mix_int(z: int) -> int:
    """splitmix64's output function on Python integers (definition)."""
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def chi2_pvalue(counts, probs):
    """Pearson chi-square p-value; cells with expected count < 5 are pooled."""
    counts = np.asarray(counts, dtype=np.float64).ravel()
    exp = np.asarray(probs, dtype=np.float64).ravel() * counts.sum()
    small = exp < 5
    if small.any():
        counts = np.append(counts[~small], counts[small].sum())
        exp = np.append(exp[~small], exp[small].sum())
        if exp[-1] == 0:
            counts, exp = counts[:-1], exp[:-1]
    stat = ((counts - exp) ** 2 / exp).sum()
    return float(scipy_stats.chi2.sf(stat, len(exp) - 1))


def test_splitmix64_published_sequence_from_state_zero():
    # splitmix64.c (S. Vigna, public domain) started from state 0 emits
    # 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4, 0x06c45d188009454f
    got = [int(x) for x in ref.rng_u64(0, 0, 0, 0, [0, 1, 2])]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_form_equals_the_sequential_generator():
    seed = 0x1234_5678_9ABC_DEF0
    state, seq = seed, []
    for _ in range(6):                       # the generator as a sequence
        state = (state + PHI) & M64
        seq.append(mix_int(state))
    assert [int(x) for x in ref.rng_u64(seed, 0, 0, 0, np.arange(6))] == seq
    # counter layout: stream << 60 | j << 52 | b << 32 | v
    for stream, j, b, v in [(3, 5, 2, 0), (1, 16, 1023, 151935), (2, 255, (1 << 20) - 1, 7)]:
        c = (stream << 60) | (j << 52) | (b << 32) | v
        assert int(ref.rng_u64(seed, stream, j, b, v)) == mix_int((seed + (c + 1) * PHI) & M64)


def test_uniforms_lie_strictly_inside_the_unit_interval_and_are_flat():
    u = ref.rng_uniform(99, 3, 0, 0, np.arange(1 << 16, dtype=np.uint64))
    assert u.min() > 0.0 and u.max() < 1.0
    assert np.all(u * (1 << 23) - 0.5 == np.floor(u * (1 << 23)))   # 23-bit grid + 1/2
    assert np.all(u.astype(np.float32).astype(np.float64) == u)      # exact in float32
    counts = np.histogram(u, bins=32, range=(0, 1))[0]
    assert chi2_pvalue(counts, np.full(32, 1 / 32)) > 1e-3


def test_gumbel_max_draws_follow_the_tempered_softmax():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal(6) * 1.5
    T = 0.7
    draws = [int(ref.draft_sample(logits[None], T, seed, 0)[0]) for seed in range(20000)]
    counts = np.bincount(draws, minlength=6)
    assert chi2_pvalue(counts, ref.softmax_t(logits, T)) > 1e-3


@pytest.mark.parametrize("seed", range(6))
def test_acceptance_plus_residual_reproduce_p_exactly(seed):
    # sum_x q(x) [ a(x) 1{y = x} + (1 - a(x)) r(y) ] = p(y): the committed
    # token is an exact draw from p whatever q is
    rng = np.random.default_rng(seed)
    V = 7
    p = ref.softmax_t(rng.standard_normal(V) * 2, 1.0)
    q = ref.softmax_t(rng.standard_normal(V) * 2, 1.0)
    r = ref.residual_distribution(p, q)
    total = np.zeros(V)
    for x in range(V):
        a = ref.accept_probability(p, q, x)
        total[x] += q[x] * a
        total += q[x] * (1 - a) * r
    np.testing.assert_allclose(total, p, rtol=0, atol=1e-12)


def test_acceptance_rate_of_the_verifier_is_min_one_p_over_q():
    rng = np.random.default_rng(11)
    V, T = 5, 1.0
    tl = rng.standard_normal((2, V))
    dl = rng.standard_normal((1, V))
    p, q = ref.softmax_t(tl[0], T), ref.softmax_t(dl[0], T)
    x = int(np.argmax(q / p))                 # a token with p(x) < q(x)
    a = ref.accept_probability(p, q, x)
    assert a < 1
    n = 20000
    acc = sum(ref.verify_sample(tl, dl, [x], T, s, 0)[0] == 2 for s in range(n))
    assert abs(acc / n - a) < 5 * np.sqrt(a * (1 - a) / n)


def test_first_committed_token_follows_the_target_distribution():
    rng = np.random.default_rng(12)
    V, T, gamma = 6, 0.8, 3
    tl = rng.standard_normal((gamma + 1, V)) * 1.5
    dl = rng.standard_normal((gamma, V)) * 1.5
    counts = np.zeros(V)
    for s in range(12000):
        d = ref.draft_sample(dl, T, s, 0)
        counts[ref.verify_sample(tl, dl, d, T, s, 0)[1][0]] += 1
    assert chi2_pvalue(counts, ref.softmax_t(tl[0], T)) > 1e-3


def test_identical_distributions_accept_everything_and_draw_the_bonus_from_p():
    rng = np.random.default_rng(13)
    V, T, gamma = 5, 1.3, 4
    tl = rng.standard_normal((gamma + 1, V))
    counts = np.zeros(V)
    for s in range(8000):
        d = ref.draft_sample(tl[:gamma], T, s, 1)
        tau, com, nxt = ref.verify_sample(tl, tl[:gamma], d, T, s, 1)
        assert tau == gamma + 1 and list(com[:gamma]) == list(d) and com[gamma] == nxt
        counts[nxt] += 1
    assert chi2_pvalue(counts, ref.softmax_t(tl[gamma], T)) > 1e-3


def test_draft_the_target_rules_out_is_always_rejected_and_replaced():
    V, T, gamma = 6, 1.0, 2
    tl = np.zeros((gamma + 1, V))
    tl[0, 4] = -1e9                           # target: token 4 impossible at row 0
    dl = np.full((gamma, V), -1e9)
    dl[:, 4] = 0.0                            # drafter: token 4 certain
    for s in range(200):
        d = ref.draft_sample(dl, T, s, 0)
        assert list(d) == [4, 4]
        tau, com, nxt = ref.verify_sample(tl, dl, d, T, s, 0)
        assert tau == 1 and com[0] != 4 and list(com[1:]) == [-1, -1]


def test_speculative_sampling_loop_is_lossless_in_distribution():
    """Two tokens after the anchor: the speculative loop with a drafter that
    knows nothing of the target (fixed random logits) reproduces the exact
    target-only sampling distribution of (y1, y2)."""
    target = sl.TinyTarget(seed=5, vocab=6, d=32, n_layers=4, n_heads=2, d_ffn=64)
    prompt, anchor, gamma, T = [1, 3, 2], 4, 3, 0.9
    table = np.random.default_rng(21).standard_normal((gamma, target.V)) * 1.2
    P = sl.target_sampling_pair_probs(target, prompt, anchor, T)
    counts = np.zeros_like(P)
    taus = []
    for s in range(3000):
        y = sl.speculative_sample_generate(target, lambda a, seq: table, prompt, anchor, 2, gamma, T,
                                           seed=1000 + s, stats=taus)
        counts[y[0], y[1]] += 1
    assert chi2_pvalue(counts, P) > 1e-3
    assert 1 <= min(taus) and max(taus) <= gamma + 1


def test_each_position_draws_its_own_acceptance_uniform():
    # keep-probability 1/2 at positions 0 and 1: both kept with probability
    # 1/4 when the positions use independent uniforms (1/2 with a shared one)
    T = 1.0
    q_logits = np.log(np.array([[0.8, 0.2], [0.8, 0.2]]))
    p_logits = np.log(np.array([[0.4, 0.6], [0.4, 0.6], [0.5, 0.5]]))
    n = 8000
    both = sum(ref.verify_sample(p_logits, q_logits, [0, 0], T, s, 0)[0] == 3 for s in range(n))
    assert abs(both / n - 0.25) < 5 * np.sqrt(0.25 * 0.75 / n)
