"""GPU parity of per-sequence block sizes (gamma_b <= gamma): sequence b's
drafts and acceptance must equal the oracle's drafting pass and verify-accept
run with gamma = gamma_b[b]."""
import dataclasses

import numpy as np
import pytest
import torch

import synth
from oracle import dflash_ref as ref
from tests import harness as H
from tests.test_gpu_parity import SMALL, planted_verify_inputs, run_chain

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dfl(lib):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return lib


@pytest.mark.parametrize("gammas", [[16, 5, 1], [1, 16, 9]])
def test_per_sequence_block_drafts_equal_the_oracle_at_that_block_size(dfl, gammas):
    lens = [300, 45, 0]
    gd = run_chain(dfl, SMALL, lens, check_dumps=False)
    wl, B = gd.wl, len(lens)
    anchors = synth.anchors(wl)
    a = torch.as_tensor(np.asarray(anchors, dtype=np.int32), device="cuda")
    gb = torch.as_tensor(np.asarray(gammas, dtype=np.int32), device="cuda")
    draft = torch.empty((B, wl.gamma), dtype=torch.int32, device="cuda")
    logits = torch.empty((B, wl.gamma, wl.vocab), dtype=torch.float32, device="cuda")
    dfl.dflash_draft_block_dyn(gd.cfg, gd.w, a, gd.ctx_len[:B], gb, max(lens), gd.k_cache, gd.v_cache, draft,
                               gd.status, gd.ws, logits=logits)
    torch.cuda.synchronize()
    gd.check_status()
    W = gd.W
    for b in range(B):
        g_b, n = gammas[b], lens[b]
        oc = dataclasses.replace(H.oracle_cfg(wl), gamma=g_b)
        # the context K/V the GPU holds (pinned to the oracle by run_chain)
        kc = [ref.f64(gd.k_cache[l, b, :, :n]) for l in range(wl.n_layers)]
        vc = [ref.f64(gd.v_cache[l, b, :, :n]) for l in range(wl.n_layers)]
        out = ref.draft_block(oc, W, int(anchors[b]), kc, vc, n)
        H.assert_logits_close(logits[b, :g_b], out["logits"], f"logits b{b} gamma_b={g_b}")
        H.assert_drafts_match(draft[b, :g_b].cpu().numpy(), out["logits"], f"draft b{b} gamma_b={g_b}")
        assert (draft[b, g_b:] == -1).all()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_per_sequence_block_verify_equals_the_oracle_at_that_block_size(dfl, dtype):
    B, V = 5, 1003
    wl = SMALL.replace(batch=B, vocab=V)
    gd = H.GpuDrafter(dfl, wl, max_rows=16, weights=synth.weights(wl, "cuda"))
    logits, draft = planted_verify_inputs(wl, dtype, seed=41)
    gammas = [16, 1, 7, 3, 12]
    gb = torch.as_tensor(np.asarray(gammas, dtype=np.int32), device="cuda")
    tau = torch.empty(B, dtype=torch.int32, device="cuda")
    committed = torch.empty((B, wl.gamma + 1), dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    dfl.dflash_verify_accept_dyn(gd.cfg, logits, torch.as_tensor(draft, device="cuda"), gb, tau, committed, nxt,
                                 gd.ws)
    torch.cuda.synchronize()
    tau, committed, nxt = tau.cpu().numpy(), committed.cpu().numpy(), nxt.cpu().numpy()
    for b in range(B):
        g_b = gammas[b]
        t, c, n = ref.verify_accept(logits[b, :g_b + 1].float().cpu(), draft[b, :g_b])
        assert tau[b] == t and nxt[b] == n, (b, tau[b], t)
        np.testing.assert_array_equal(committed[b, :g_b + 1], c)
        assert (committed[b, g_b + 1:] == -1).all()
    # gamma_b = gamma everywhere is plain verify-accept
    full = torch.full((B,), wl.gamma, dtype=torch.int32, device="cuda")
    d = torch.as_tensor(draft, device="cuda")
    tau2 = torch.empty(B, dtype=torch.int32, device="cuda")
    c2 = torch.empty((B, wl.gamma + 1), dtype=torch.int32, device="cuda")
    n2 = torch.empty(B, dtype=torch.int32, device="cuda")
    dfl.dflash_verify_accept_dyn(gd.cfg, logits, d, full, tau2, c2, n2, gd.ws)
    t3, c3, n3 = gd.verify(logits, d)
    torch.cuda.synchronize()
    assert torch.equal(tau2, t3) and torch.equal(c2, c3) and torch.equal(n2, n3)
