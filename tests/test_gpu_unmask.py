"""GPU parity of multi-step confidence unmasking: every pass on the GPU's
block ids against the oracle's pass on the same ids, every unmasking decision
against the oracle's, and the one-call multi-pass API against the composition
of its steps."""
import numpy as np
import pytest
import torch

import synth
from oracle import dflash_ref as ref
from tests import harness as H
from tests.test_gpu_parity import SMALL, run_chain

pytestmark = pytest.mark.gpu

CONF_TIE = 1e-4   # relative confidence gap below which fp32 and fp64 may pick differently


@pytest.fixture(scope="module")
def dfl(lib):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return lib


def check_decision(gpu_ids, ids, oracle_logits, steps_left, mask_id, what):
    """GPU decision equals the oracle's, or differs only inside a confidence tie."""
    want = ref.unmask_step(ids, oracle_logits, steps_left, mask_id)
    if np.array_equal(gpu_ids, want):
        return 0
    conf = ref.confidence(oracle_logits)
    tok = ref.argmax_lowest(ref.f64(oracle_logits))
    picked_g = {j for j in range(len(conf)) if ids[j + 1] == mask_id and gpu_ids[j + 1] != mask_id}
    picked_o = {j for j in range(len(conf)) if ids[j + 1] == mask_id and want[j + 1] != mask_id}
    assert len(picked_g) == len(picked_o), what
    for j in picked_g:   # the GPU's tokens are the pass's argmax tokens (ties excepted by the logit rule)
        assert gpu_ids[j + 1] == tok[j] or abs(np.sort(ref.f64(oracle_logits)[j])[-1]
                                               - np.sort(ref.f64(oracle_logits)[j])[-2]) < H.MARGIN, what
    lo = min(conf[j] for j in picked_g)
    hi = max(conf[j] for j in picked_o - picked_g) if picked_o - picked_g else lo
    assert abs(hi - lo) <= CONF_TIE * hi, (what, sorted(picked_g), sorted(picked_o), lo, hi)
    return 1


@pytest.mark.parametrize("n_steps", [4, 16])
def test_unmasking_passes_and_decisions_follow_the_oracle(dfl, n_steps):
    lens = [300, 45, 0]
    gd = run_chain(dfl, SMALL, lens, check_dumps=False)
    wl, B, R, m = gd.wl, len(lens), gd.wl.rows, gd.wl.vocab - 1
    anchors = synth.anchors(wl)
    kc = [[ref.f64(gd.k_cache[l, b, :, :lens[b]]) for l in range(wl.n_layers)] for b in range(B)]
    vc = [[ref.f64(gd.v_cache[l, b, :, :lens[b]]) for l in range(wl.n_layers)] for b in range(B)]
    oc = H.oracle_cfg(wl)
    ids = torch.full((B, R), m, dtype=torch.int32, device="cuda")
    ids[:, 0] = torch.as_tensor(np.asarray(anchors, dtype=np.int32))
    draft = torch.empty((B, wl.gamma), dtype=torch.int32, device="cuda")
    logits = torch.empty((B, wl.gamma, wl.vocab), dtype=torch.float32, device="cuda")
    ties = 0
    for s in range(n_steps):
        before = ids.cpu().numpy().copy()
        dfl.dflash_draft_block_ids(gd.cfg, gd.w, ids, gd.ctx_len[:B], max(lens), gd.k_cache, gd.v_cache, draft,
                                   gd.status, gd.ws, logits=logits)
        dfl.dflash_unmask_step(gd.cfg, logits, draft, ids, n_steps - s, gd.ws)
        torch.cuda.synchronize()
        gd.check_status()
        after = ids.cpu().numpy()
        for b in range(B):
            out = ref.draft_block(oc, gd.W, int(anchors[b]), kc[b], vc[b], lens[b], ids=before[b])
            H.assert_logits_close(logits[b], out["logits"], f"pass {s} logits b{b}")
            ties += check_decision(after[b], before[b], out["logits"], n_steps - s, m, f"pass {s} b{b}")
    assert (ids[:, 1:] != m).all()
    H.report(f"unmask {n_steps} passes", "decisions differing at confidence ties", ties, 0)


def test_multi_pass_call_is_the_composition_of_its_steps(dfl):
    lens = [300, 45, 0]
    gd = run_chain(dfl, SMALL, lens, check_dumps=False)
    wl, B, R, m = gd.wl, len(lens), gd.wl.rows, gd.wl.vocab - 1
    a = torch.as_tensor(np.asarray(synth.anchors(wl), dtype=np.int32), device="cuda")
    logits = torch.empty((B, wl.gamma, wl.vocab), dtype=torch.float32, device="cuda")
    for n_steps in (1, 5):
        ids = torch.empty((B, R), dtype=torch.int32, device="cuda")
        draft = torch.empty((B, wl.gamma), dtype=torch.int32, device="cuda")
        dfl.dflash_draft_block_iter(gd.cfg, gd.w, a, gd.ctx_len[:B], max(lens), gd.k_cache, gd.v_cache, n_steps,
                                    ids, draft, logits, gd.status, gd.ws)
        # the same steps composed by hand
        ids2 = torch.full((B, R), m, dtype=torch.int32, device="cuda")
        ids2[:, 0] = a
        d2 = torch.empty_like(draft)
        for s in range(n_steps):
            dfl.dflash_draft_block_ids(gd.cfg, gd.w, ids2, gd.ctx_len[:B], max(lens), gd.k_cache, gd.v_cache, d2,
                                       gd.status, gd.ws, logits=logits)
            dfl.dflash_unmask_step(gd.cfg, logits, d2, ids2, n_steps - s, gd.ws)
        torch.cuda.synchronize()
        gd.check_status()
        assert torch.equal(ids, ids2) and torch.equal(draft, ids2[:, 1:])
        if n_steps == 1:   # one pass is the single-pass draft
            greedy, _, _ = gd.draft(synth.anchors(wl), max(lens))
            assert torch.equal(draft, greedy)
