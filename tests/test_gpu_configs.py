"""GPU parity at the full workload sizes: long context (N = 32768), the ragged
batch of 16 sequences, the multi-cycle draft-verify loop, and the device-side
capacity error. Context K/V is filled directly with synthetic bf16 rows
(both sides read the same values) where recomputing it in the oracle would
take minutes; fusion and injection are compared on sampled rows, each of
which the oracle computes independently."""
import numpy as np
import pytest
import torch

import synth
from oracle import dflash_ref as ref
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dfl(lib):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return lib


def f64_weights(W):
    """Weights as float64 once (the oracle accepts any array; this only saves
    repeated conversion across many oracle calls). The embedding stays a tensor."""
    return {k: (v.cpu() if k == "embed" else ref.f64(v)) for k, v in W.items()}


def fill_cache(gd, lens, tag):
    """Context rows 0..len-1 of every (layer, sequence, kv head) from synth."""
    wl = gd.wl
    n = int(max(lens))
    k = synth.kv_rows(wl, n, tag + "/k", "cuda")
    v = synth.kv_rows(wl, n, tag + "/v", "cuda")
    for b, nb in enumerate(lens):
        gd.k_cache[:, b, :, :nb] = k[:, b, :, :nb]
        gd.v_cache[:, b, :, :nb] = v[:, b, :, :nb]
    gd.ctx_len[: len(lens)] = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    return k, v


def check_draft(gd, W64, anchors, lens, k, v, seqs):
    oc = H.oracle_cfg(gd.wl)
    draft, logits, _ = gd.draft(anchors, int(max(lens)), want_logits=True)
    torch.cuda.synchronize()
    gd.check_status()
    for b in seqs:
        nb = int(lens[b])
        kc = [ref.f64(k[l, b, :, :nb]) for l in range(gd.wl.n_layers)]
        vc = [ref.f64(v[l, b, :, :nb]) for l in range(gd.wl.n_layers)]
        out = ref.draft_block(oc, W64, int(anchors[b]), kc, vc, nb)
        H.assert_logits_close(logits[b], out["logits"], f"logits b{b} n={nb}")
        H.assert_drafts_match(draft[b].cpu().numpy(), out["logits"], f"draft b{b} n={nb}")


def check_fuse_inject_rows(gd, W64, taps, n_rows, sample, pos0=0):
    """ctx_fuse + kv_inject of n_rows rows of sequence 0 on the GPU; the oracle
    recomputes the sampled rows (rows are independent)."""
    oc = H.oracle_cfg(gd.wl)
    h = gd.fuse(taps)
    gd.inject(h.view(1, n_rows, -1), [n_rows])
    torch.cuda.synchronize()
    gd.check_status()
    idx = np.asarray(sample)
    h_or = ref.ctx_fuse(oc, W64["w_c"], W64["g_c"], taps[idx].float().cpu())
    H.assert_act_close(h[idx], h_or, "H_t sampled rows")
    for l in range(gd.wl.n_layers):
        kk, vv = ref.ctx_kv(oc, W64["w_qkv"][l], h_or, 0, positions=pos0 + idx)
        H.assert_act_close(gd.k_cache[l, 0, :, pos0 + idx], kk, f"K rows l{l}")
        H.assert_act_close(gd.v_cache[l, 0, :, pos0 + idx], vv, f"V rows l{l}")


def test_long_context_n32768(dfl):
    wl = synth.WORKLOADS["qwen3_8b_L5_N32768_B1"]
    gd = H.GpuDrafter(dfl, wl, max_rows=wl.ctx)
    W64 = f64_weights(gd.W)
    # fusion + injection over the whole long prefill, sampled rows (ragged tail included)
    taps = synth.taps(wl, wl.ctx, "prefill", "cuda")
    rng = np.random.default_rng(5)
    sample = np.unique(np.concatenate([[0, 1, 127, 128, wl.ctx - 1], rng.integers(0, wl.ctx, 27)]))
    check_fuse_inject_rows(gd, W64, taps, wl.ctx, sample)
    del taps
    # the draft block over a directly filled 32768-row context
    lens = [wl.ctx]
    k, v = fill_cache(gd, lens, "c3")
    check_draft(gd, W64, synth.anchors(wl), lens, k, v, [0])


def test_ragged_batch_16(dfl):
    wl = synth.WORKLOADS["qwen3_8b_L5_ragged_B16"]
    lens = synth.ctx_lengths(wl)
    gd = H.GpuDrafter(dfl, wl, max_rows=16)
    W64 = f64_weights(gd.W)
    k, v = fill_cache(gd, lens, "c4")
    check_draft(gd, W64, synth.anchors(wl), lens, k, v, range(wl.batch))


def test_capacity_overflow_sets_status_and_skips(dfl):
    wl = synth.Workload("cap_bf16", n_layers=1, d_target=128, n_taps=5, d_model=256, n_q_heads=8,
                        n_kv_heads=2, head_dim=128, d_ffn=384, vocab=1003, gamma=16, dtype="bf16",
                        batch=2, ctx=64, seed=31)
    gd = H.GpuDrafter(dfl, wl, max_rows=64, ctx_capacity=64)
    h = synth.hidden(wl, 2 * 60, "cap", "cuda").view(2, 60, -1)
    # sequence 0: 40 rows fit (40 <= 64 - 17); sequence 1: 60 rows do not
    gd.inject(h, [40, 60])
    torch.cuda.synchronize()
    assert int(gd.status.item()) == dfl.ERR_CAPACITY
    assert gd.ctx_len[:2].cpu().tolist() == [40, 0]
    assert float(gd.k_cache[0, 1].abs().sum()) == 0.0        # nothing written for sequence 1
    assert float(gd.k_cache[0, 0, :, :40].abs().sum()) > 0.0


def test_draft_verify_loop_8_layers(dfl):
    """All 256 cycles of the 8-layer batch-4 loop (context 4096 growing by tau
    every cycle) on the GPU, the oracle teacher-forced on the GPU's state.

    Every cycle: the synthetic target's logits are made from the GPU's drafts
    (it agrees with a drafted token with probability 0.8, decided by a hash of
    the token itself, so a wrong draft changes the acceptance pattern), and
    the oracle's verify-accept on those drafts must give the GPU's tau,
    committed tokens and next anchor exactly. At a seeded sample of cycles
    (the first two, the last, and four others) the oracle also drafts from the
    GPU's anchor and its context K/V at that cycle (logits within tolerance,
    drafts equal outside near-ties) and recomputes the rows injected in that
    cycle (fusion of the accepted positions' tapped states, K/V of every
    layer at their positions). One near-tie therefore cannot derail later
    comparisons."""
    wl = synth.WORKLOADS["qwen3_8b_L8_loop_B4"]
    B, R, L = wl.batch, wl.rows, wl.n_layers
    lens = synth.ctx_lengths(wl)
    gd = H.GpuDrafter(dfl, wl, max_rows=B * R)
    W64 = f64_weights(gd.W)
    oc = H.oracle_cfg(wl)
    k, v = fill_cache(gd, lens, "c5")
    del k, v
    rng = np.random.default_rng(5005)
    sample = {0, 1, wl.cycles - 1} | {int(c) for c in rng.choice(np.arange(2, wl.cycles - 1), 4, replace=False)}
    anchor = torch.as_tensor(synth.anchors(wl), device="cuda")
    draft = torch.empty((B, wl.gamma), dtype=torch.int32, device="cuda")
    logits = torch.empty((B, wl.gamma, wl.vocab), dtype=torch.float32, device="cuda")
    taus, draft_checks, agree_changed = [], 0, 0
    total = np.asarray(lens, dtype=np.int64).copy()
    for cyc in range(wl.cycles):
        check = cyc in sample
        len_before = gd.ctx_len[:B].cpu().numpy().copy()
        anchor_before = anchor.cpu().numpy().copy()
        gd.lib.dflash_draft_block(gd.cfg, gd.w, anchor, gd.ctx_len[:B], wl.ctx + cyc * R, gd.k_cache,
                                  gd.v_cache, draft, gd.status, gd.ws, logits=logits if check else None)
        tl = synth.loop_target_logits(wl, cyc, draft)
        tau, committed, nxt = gd.verify(tl, draft)
        taps = synth.taps(wl, B * R, f"loop{cyc}", "cuda")
        h = gd.fuse(taps).view(B, R, -1)
        gd.lib.dflash_kv_inject(gd.cfg, gd.w, h, tau, gd.ctx_len[:B], gd.k_cache, gd.v_cache,
                                gd.status, gd.ws)
        torch.cuda.synchronize()
        gd.check_status()
        d_np, tl_np = draft.cpu().numpy(), tl.cpu().numpy()
        tau_np, com_np, nxt_np = tau.cpu().numpy(), committed.cpu().numpy(), nxt.cpu().numpy()
        # the agreement pattern depends on the drafted tokens themselves
        key16, offset = synth.loop_plan(wl, cyc)
        alt = synth.loop_intended(wl, torch.as_tensor(key16), torch.as_tensor(offset),
                                  torch.as_tensor((d_np + 1) % wl.vocab))
        now = synth.loop_intended(wl, torch.as_tensor(key16), torch.as_tensor(offset), torch.as_tensor(d_np))
        agree_changed += int(((alt[:, :-1] == torch.as_tensor((d_np + 1) % wl.vocab)) !=
                              (now[:, :-1] == torch.as_tensor(d_np))).sum())
        for b in range(B):
            t, c, n = ref.verify_accept(tl_np[b], d_np[b])
            assert int(tau_np[b]) == t, (cyc, b, int(tau_np[b]), t)
            assert com_np[b].tolist() == c.tolist(), (cyc, b)
            assert int(nxt_np[b]) == n, (cyc, b)
            taus.append(t)
            total[b] += t
        if check:
            for b in range(B):
                nb = int(len_before[b])
                kc = [ref.f64(gd.k_cache[l, b, :, :nb]) for l in range(L)]
                vc = [ref.f64(gd.v_cache[l, b, :, :nb]) for l in range(L)]
                out = ref.draft_block(oc, W64, int(anchor_before[b]), kc, vc, nb)
                del kc, vc
                H.assert_logits_close(logits[b], out["logits"], f"cycle {cyc} logits b{b}")
                H.assert_drafts_match(d_np[b], out["logits"], f"cycle {cyc} draft b{b}", gpu_logits=logits[b])
                draft_checks += 1
                t = int(tau_np[b])
                h_or = ref.ctx_fuse(oc, W64["w_c"], W64["g_c"], taps.view(B, R, -1)[b, :t].float().cpu())
                H.assert_act_close(h[b, :t], h_or, f"cycle {cyc} H_t b{b}")
                for l in range(L):
                    kk, vv = ref.ctx_kv(oc, W64["w_qkv"][l], h_or, nb)
                    H.assert_act_close(gd.k_cache[l, b, :, nb:nb + t], kk, f"cycle {cyc} K rows l{l} b{b}")
                    H.assert_act_close(gd.v_cache[l, b, :, nb:nb + t], vv, f"cycle {cyc} V rows l{l} b{b}")
        anchor = nxt.clone()
        assert gd.ctx_len[:B].cpu().tolist() == total.tolist()
    assert all(1 <= t <= R for t in taus)
    assert draft_checks == len(sample) * B
    assert agree_changed > 0        # a different token would have changed some decisions
    mean_tau = float(np.mean(taus))
    assert 4.0 < mean_tau < 6.0, mean_tau   # E[tau] = 4.89 for agreement probability 0.8
    H.report("loop", "teacher-forced draft checks", draft_checks, 0)
    H.report("loop", "mean tau", mean_tau, 0)
