"""GPU parity: the C-ABI path against the CPU oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import synth
from oracle import dflash_ref as ref
from tests import harness as H

pytestmark = pytest.mark.gpu

SMALL = synth.Workload("small_bf16_L2", n_layers=2, d_target=128, n_taps=5, d_model=256,
                       n_q_heads=8, n_kv_heads=2, head_dim=128, d_ffn=384, vocab=1003, gamma=16,
                       dtype="bf16", batch=3, ctx=300, seed=7)


@pytest.fixture(scope="module")
def dfl(lib):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return lib


# ------------------------------------------------------------------ projection unit

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (17, 384, 256), (100, 256, 4096),
                                   (272, 640, 512), (600, 384, 1024), (2048, 1024, 512),
                                   (33, 4096, 4096),
                                   # token-major tiles whose feature count is not a multiple of
                                   # 16 (scalar stores) or of the 256-feature tile (a ragged last tile)
                                   (700, 200, 256), (1030, 600, 320)])
def test_linear_matches_fp32_matmul(dfl, dtype, M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M * 7919 + N * 31 + K)
    x = torch.randn((M, K), generator=g, device="cuda").to(dtype)
    w = (torch.randn((N, K), generator=g, device="cuda") / K ** 0.5).to(dtype)
    y = torch.full((M, N), float("nan"), device="cuda")
    cfg = dfl.config_from_workload(SMALL)
    ws = dfl.Workspace(cfg, 16)
    dfl.dflash_linear(x, w, y, ws)
    torch.cuda.synchronize()
    want = x.double() @ w.double().T
    err = (y.double() - want).abs().max().item()
    rms = want.pow(2).mean().sqrt().item()
    tol = 1e-4 if dtype == torch.bfloat16 else 5e-3   # fp32 inputs run as tf32
    assert err <= tol * rms * 10, (err, rms)


# ------------------------------------------------------------------ verify-accept

def planted_verify_inputs(wl, dtype, seed):
    B, R, V = wl.batch, wl.rows, wl.vocab
    logits = synth.target_logits(wl, f"verify{seed}", "cuda", torch.float32)
    rng = np.random.default_rng(seed)
    draft = rng.integers(0, V, size=(B, wl.gamma)).astype(np.int32)
    for b in range(B):
        k = [0, wl.gamma, 1, 5, 9][b % 5]         # planted accepted prefix length
        for j in range(k):
            row = logits[b, j]
            row[int(draft[b, j])] = row.max() + 1.0
        if b % 3 == 2:                              # a tie at the bonus row: lowest index wins
            row = logits[b, k]
            top = row.max() + 2.0
            i1, i2 = sorted(rng.choice(V, size=2, replace=False))
            row[int(i1)] = top
            row[int(i2)] = top
    return logits.to(dtype), draft


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,V", [(1, 151936), (5, 1003), (7, 4096)])
def test_verify_accept_bit_exact(dfl, dtype, B, V):
    wl = SMALL.replace(batch=B, vocab=V)
    gd = H.GpuDrafter(dfl, wl, max_rows=16, weights={k: v for k, v in synth.weights(SMALL.replace(vocab=V), "cuda").items()})
    logits, draft = planted_verify_inputs(wl, dtype, seed=B * 100 + V % 97)
    tau, committed, nxt = gd.verify(logits, torch.as_tensor(draft, device="cuda"))
    tau, committed, nxt = tau.cpu().numpy(), committed.cpu().numpy(), nxt.cpu().numpy()
    for b in range(B):
        t, c, n = ref.verify_accept(logits[b].float().cpu(), draft[b])
        assert tau[b] == t and nxt[b] == n, (b, tau[b], t)
        np.testing.assert_array_equal(committed[b], c)
    # repeated calls reuse the workspace counters: same answer again
    tau2, committed2, _ = gd.verify(logits, torch.as_tensor(draft, device="cuda"))
    np.testing.assert_array_equal(tau2.cpu().numpy(), tau)
    np.testing.assert_array_equal(committed2.cpu().numpy(), committed)


# ------------------------------------------------------------------ full chain

def run_chain(dfl, wl, ctx_lens, check_dumps=True, max_rows=None):
    """taps -> ctx_fuse -> kv_inject -> draft_block on the GPU and in the oracle."""
    B = len(ctx_lens)
    total = int(sum(ctx_lens))
    gd = H.GpuDrafter(dfl, wl, max_rows=max(max_rows or 0, total, 16))
    oc = H.oracle_cfg(wl)
    taps = synth.taps(wl, max(total, 1), "ctx", "cuda")[:total]
    h_gpu = gd.fuse(taps) if total else torch.empty((0, wl.d_model), dtype=gd.dt, device="cuda")
    tmax = max(max(ctx_lens), 1)
    h_pad = torch.zeros((B, tmax, wl.d_model), dtype=gd.dt, device="cuda")
    offs = np.concatenate([[0], np.cumsum(ctx_lens)])
    for b in range(B):
        h_pad[b, : ctx_lens[b]] = h_gpu[offs[b]:offs[b + 1]]
    gd.inject(h_pad, ctx_lens)
    torch.cuda.synchronize()
    gd.check_status()
    assert gd.ctx_len[:B].cpu().tolist() == list(ctx_lens)

    k_all = gd.k_cache.clone()
    v_all = gd.v_cache.clone()
    anchors = synth.anchors(wl)
    draft, logits, dump = gd.draft(anchors, max(ctx_lens), want_logits=True, want_dump=check_dumps)
    # without a logits copy the LM head's argmax takes its other epilogue
    # (one thread per token): the same drafts bit for bit
    draft_nl, _, _ = gd.draft(anchors, max(ctx_lens))
    torch.cuda.synchronize()
    gd.check_status()
    assert torch.equal(draft_nl, draft)

    W = gd.W
    for b in range(B):
        n = ctx_lens[b]
        taps_b = taps[offs[b]:offs[b + 1]]
        h_or = ref.ctx_fuse(oc, W["w_c"], W["g_c"], taps_b.float().cpu()) if n else np.zeros((0, wl.d_model))
        if n:
            H.assert_act_close(h_gpu[offs[b]:offs[b + 1]], h_or, f"H_t[{b}]")
        kc, vc = [], []
        for l in range(wl.n_layers):
            k, v = ref.ctx_kv(oc, W["w_qkv"][l], h_or, 0)
            kc.append(k)
            vc.append(v)
            if n:
                H.assert_act_close(k_all[l, b, :, :n], k, f"K cache l{l} b{b}")
                H.assert_act_close(v_all[l, b, :, :n], v, f"V cache l{l} b{b}")
        out = ref.draft_block(oc, W, int(anchors[b]), kc, vc, n, want_dumps=check_dumps)
        if check_dumps:
            R = wl.rows
            for l in range(wl.n_layers + 1):
                H.assert_act_close(dump[l, b * R:(b + 1) * R], out["dumps"][l], f"h after layer {l} b{b}")
        H.assert_logits_close(logits[b], out["logits"], f"logits b{b}")
        H.assert_drafts_match(draft[b].cpu().numpy(), out["logits"], f"draft b{b}")
    return gd


def test_chain_small_bf16_ragged_batch(dfl):
    run_chain(dfl, SMALL, [300, 45, 0])


def test_chain_small_bf16_long_prefill_plain_gemm(dfl):
    # > 512 fused rows: context fusion / injection take the token-major GEMM
    run_chain(dfl, SMALL.replace(batch=2, ctx=700), [700, 513])


def test_chain_bf16_d384_prefill_half_valid_feature_tile(dfl):
    # D = 384: the token-major fusion tiles are 256 features wide, so the
    # second tile has 128 valid features (its sums of squares and stores
    # must stop at D); Dh = 64 heads: four per 256-feature injection tile
    wl = synth.Workload("d384_bf16", n_layers=1, d_target=128, n_taps=5, d_model=384, n_q_heads=6,
                        n_kv_heads=2, head_dim=64, d_ffn=512, vocab=1003, gamma=16, dtype="bf16",
                        batch=2, ctx=600, seed=13)
    run_chain(dfl, wl, [600, 77])


def test_chain_small_bf16_rope_off(dfl):
    run_chain(dfl, SMALL.replace(rope_theta=0.0, batch=1), [130])


def test_chain_small_bf16_vocab_over_1280_tiles(dfl):
    # 200003 entries = 1563 LM-head tiles (the last one 67 rows): the per-token
    # reduction of the tiles' argmax keys takes more than one pass of its CTA
    run_chain(dfl, SMALL.replace(n_layers=1, batch=2, vocab=200003), [64, 9], check_dumps=False)


MEDIUM = synth.Workload("medium_bf16_L2", n_layers=2, d_target=512, n_taps=5, d_model=1024,
                        n_q_heads=8, n_kv_heads=2, head_dim=128, d_ffn=2048, vocab=5000, gamma=16,
                        dtype="bf16", batch=2, ctx=1000, seed=9)


def test_chain_medium_bf16_split_k_clusters(dfl):
    # K = 1024..2560 gives 4-8 k-splits per projection: exercises the cluster reduction
    run_chain(dfl, MEDIUM, [1000, 77])


def test_chain_medium_bf16_gamma_8(dfl):
    run_chain(dfl, MEDIUM.replace(gamma=8, batch=3, ctx=400), [400, 1, 250])


def test_chain_tiny_f32(dfl):
    wl = synth.WORKLOADS["tiny_f32_L1_N128"]
    run_chain(dfl, wl, [wl.ctx])


def test_chain_qwen3_8b_N2048(dfl):
    wl = synth.WORKLOADS["qwen3_8b_L5_N2048_B1"]
    run_chain(dfl, wl, [wl.ctx], check_dumps=True)


def test_chain_small_bf16_batch_32_several_token_tiles(dfl):
    # 32 sequences x 17 rows = 544 block rows: every drafting projection takes
    # three 256-row token tiles (the last one 32 rows), the LM head one
    # 512-row tile; ragged contexts, some empty
    lens = [int(x) for x in np.random.default_rng(32).integers(0, 160, size=32)]
    lens[3] = 0
    run_chain(dfl, SMALL.replace(n_layers=1, batch=32, ctx=160), lens, check_dumps=True)


def test_chain_small_bf16_batch_72_beyond_longest_first_order(dfl):
    # 72 x 17 = 1224 block rows: every drafting projection takes five 256-row
    # token tiles; more sequences than the attention's longest-context-first
    # mapping of launch slots covers (64), so the slots keep launch order;
    # ragged contexts, some empty, some equal
    lens = [int(x) for x in np.random.default_rng(72).integers(0, 96, size=72)]
    lens[5] = 0
    lens[40] = lens[41]
    run_chain(dfl, SMALL.replace(n_layers=1, batch=72, ctx=96), lens, check_dumps=False)


def test_chain_medium_bf16_batch_40_lm_head_several_tiles(dfl):
    # 40 x 17 = 680 block rows and 640 mask rows: the LM head's token rows
    # span three tiles too; K = 1024..2048 splits the projections over clusters
    lens = [int(x) for x in np.random.default_rng(40).integers(1, 90, size=40)]
    run_chain(dfl, MEDIUM.replace(n_layers=1, batch=40, ctx=90), lens, check_dumps=False)
