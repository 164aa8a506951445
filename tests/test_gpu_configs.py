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
    """Six cycles of the 8-layer batch-4 loop, GPU and oracle each running
    their own loop from the same inputs (device-side tau feeds the GPU's next
    injection and anchor without a host round trip).

    The acceptance pattern of the synthetic target is seeded, so tau and the
    context lengths are token-independent and must match every cycle for
    every sequence. Drafts, committed tokens and the next anchor must match
    bit-exactly (drafts: near-ties excepted) while a sequence is in step; a
    near-tie that changes the rejected position's token changes that
    sequence's next anchor, after which only its tau and length are compared."""
    wl = synth.WORKLOADS["qwen3_8b_L8_loop_B4"].replace(cycles=6)
    B, R = wl.batch, wl.rows
    lens = synth.ctx_lengths(wl)
    gd = H.GpuDrafter(dfl, wl, max_rows=B * R)
    W64 = f64_weights(gd.W)
    oc = H.oracle_cfg(wl)
    k, v = fill_cache(gd, lens, "c5")
    ok_k = [[ref.f64(k[l, b, :, : lens[b]]) for l in range(wl.n_layers)] for b in range(B)]
    ok_v = [[ref.f64(v[l, b, :, : lens[b]]) for l in range(wl.n_layers)] for b in range(B)]
    del k, v
    o_len = [int(x) for x in lens]
    g_anchor = torch.as_tensor(synth.anchors(wl), device="cuda")
    o_anchor = [int(x) for x in synth.anchors(wl)]
    in_step = [True] * B
    token_checks, taus = 0, []
    for cyc in range(wl.cycles):
        draft, logits, _ = gd.draft(g_anchor.cpu().numpy(), max(o_len) + R, want_logits=True)
        tl = synth.loop_target_logits(wl, cyc, draft)
        tau, committed, nxt = gd.verify(tl, draft)
        taps = synth.taps(wl, B * R, f"loop{cyc}", "cuda")
        h = gd.fuse(taps).view(B, R, -1)
        gd.lib.dflash_kv_inject(gd.cfg, gd.w, h, tau, gd.ctx_len[:B], gd.k_cache, gd.v_cache,
                                gd.status, gd.ws)
        g_anchor = nxt
        torch.cuda.synchronize()
        gd.check_status()
        for b in range(B):
            out = ref.draft_block(oc, W64, o_anchor[b], ok_k[b], ok_v[b], o_len[b])
            o_tl = synth.loop_target_logits(wl, cyc, torch.as_tensor(out["draft"][None]), seqs=[b])[0]
            t, c, n = ref.verify_accept(o_tl.numpy(), out["draft"])
            assert int(tau[b]) == t, (cyc, b, int(tau[b]), t)
            if in_step[b]:
                nd = H.assert_drafts_match(draft[b].cpu().numpy(), out["logits"], f"cycle {cyc} b{b}",
                                           gpu_logits=logits[b])
                token_checks += 1
                if nd == 0:
                    assert committed[b].cpu().tolist() == c.tolist()
                    assert int(nxt[b]) == n
                elif int(nxt[b]) != n:
                    in_step[b] = False
            h_or = ref.ctx_fuse(oc, W64["w_c"], W64["g_c"], taps.view(B, R, -1)[b, :t].float().cpu())
            for l in range(wl.n_layers):
                kk, vv = ref.ctx_kv(oc, W64["w_qkv"][l], h_or, o_len[b])
                ok_k[b][l] = np.concatenate([ok_k[b][l], kk], axis=1)
                ok_v[b][l] = np.concatenate([ok_v[b][l], vv], axis=1)
            o_len[b] += t
            o_anchor[b] = n
            taus.append(t)
        assert gd.ctx_len[:B].cpu().tolist() == o_len
    assert all(1 <= t <= R for t in taus)
    H.report("loop", "token-level cycle checks", token_checks, 0)
    H.report("loop", "mean tau", float(np.mean(taus)), 0)
    assert token_checks >= B
