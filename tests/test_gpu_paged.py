"""GPU parity of the paged KV cache against the oracle: the rows injected
through a page table equal the oracle's K/V (RoPE at each row's position)
within the activation tolerance, and the paged drafting pass gives the
oracle's logits and drafts, wherever the pages sit in the pool. The paged
results also equal the contiguous cache's bit for bit, and a missing page is
a capacity error."""
import numpy as np
import pytest
import torch

import synth
from oracle import dflash_ref as ref
from tests import harness as H
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu

PAGE = 128


@pytest.fixture(scope="module")
def dfl(lib):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return lib


def page_view(dfl, wl, pages_per_seq, n_pages, seed, holes=()):
    """Pools [L, n_pages, Hkv, 128, Dh] and a scrambled page table."""
    rng = np.random.default_rng(seed)
    table = rng.permutation(n_pages)[: wl.batch * pages_per_seq].reshape(wl.batch, pages_per_seq)
    for b, i in holes:
        table[b, i] = -1
    shape = (wl.n_layers, n_pages, wl.n_kv_heads, PAGE, wl.head_dim)
    dt = synth.torch_dtype(wl.dtype)
    k_pool = torch.zeros(shape, dtype=dt, device="cuda")
    v_pool = torch.zeros(shape, dtype=dt, device="cuda")
    t = torch.as_tensor(table.astype(np.int32), device="cuda")
    return dfl.KvPages(k_pool, v_pool, t), table, k_pool, v_pool


def fused_context(gd, lens, with_taps=False):
    wl = gd.wl
    total = int(sum(lens))
    taps = synth.taps(wl, total, "ctx", "cuda")
    h = gd.fuse(taps)
    h_pad = torch.zeros((len(lens), max(lens), wl.d_model), dtype=gd.dt, device="cuda")
    offs = np.concatenate([[0], np.cumsum(lens)])
    for b in range(len(lens)):
        h_pad[b, : lens[b]] = h[offs[b]:offs[b + 1]]
    if with_taps:
        return h_pad, [taps[offs[b]:offs[b + 1]] for b in range(len(lens))]
    return h_pad


def oracle_context(gd, taps_b):
    """The oracle's fused context and per-layer K/V of one sequence."""
    oc = H.oracle_cfg(gd.wl)
    n = taps_b.shape[0]
    h_or = (ref.ctx_fuse(oc, gd.W["w_c"], gd.W["g_c"], taps_b.float().cpu()) if n
            else np.zeros((0, gd.wl.d_model)))
    kv = [ref.ctx_kv(oc, gd.W["w_qkv"][l], h_or, 0) for l in range(gd.wl.n_layers)]
    return [k for k, _ in kv], [v for _, v in kv]


LENS = {3: [300, 45, 0], 2: [200, 9], 5: [60, 33, 0, 17, 50]}


# batch 5: 300 injected rows and 85 block rows, so that injection and the
# block's Q/K/V projection take the decode GEMM's wide-tile epilogues
@pytest.mark.parametrize("wl", [SMALL, SMALL.replace(batch=5, ctx=60),
                                synth.WORKLOADS["tiny_f32_L1_N128"].replace(batch=2)],
                         ids=["bf16_tcgen05", "bf16_wide_tiles", "fp32_simt"])
def test_paged_cache_matches_the_oracle_and_the_contiguous_cache(dfl, wl):
    lens = LENS[wl.batch]
    cap = 512
    gd = H.GpuDrafter(dfl, wl, max_rows=max(sum(lens), 16), ctx_capacity=cap)
    B = wl.batch
    h_pad, taps = fused_context(gd, lens, with_taps=True)
    gd.inject(h_pad, lens)
    n_new = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    anchors = synth.anchors(wl)
    a = torch.as_tensor(np.asarray(anchors, dtype=np.int32), device="cuda")
    draft_c, logits_c, _ = gd.draft(anchors, max(lens), want_logits=True)
    torch.cuda.synchronize()
    gd.check_status()
    oc = H.oracle_cfg(wl)
    want = []       # per sequence: the oracle's context K/V and its draft over them
    for b in range(B):
        kc, vc = oracle_context(gd, taps[b])
        want.append((kc, vc, ref.draft_block(oc, gd.W, int(anchors[b]), kc, vc, lens[b])))
    for seed in (1, 2):   # two different placements of the pages in the pool
        pages, table, k_pool, v_pool = page_view(dfl, wl, cap // PAGE, B * cap // PAGE + 5, seed)
        ctx2 = torch.zeros(B, dtype=torch.int32, device="cuda")
        dfl.dflash_kv_inject_paged(gd.cfg, gd.w, h_pad, n_new, ctx2, pages, gd.status, gd.ws)
        torch.cuda.synchronize()
        gd.check_status()
        assert ctx2.cpu().tolist() == list(lens)
        for b in range(B):
            kc, vc, _ = want[b]
            for p0 in range(0, lens[b], PAGE):
                n = min(PAGE, lens[b] - p0)
                pg = int(table[b, p0 // PAGE])
                for l in range(wl.n_layers):
                    # the page's rows against the oracle's K/V at positions p0 .. p0+n-1
                    H.assert_act_close(k_pool[l, pg, :, :n], kc[l][:, p0:p0 + n], f"paged K l{l} b{b} p{p0}")
                    H.assert_act_close(v_pool[l, pg, :, :n], vc[l][:, p0:p0 + n], f"paged V l{l} b{b} p{p0}")
                assert torch.equal(k_pool[:, pg, :, :n], gd.k_cache[:, b, :, p0:p0 + n])
                assert torch.equal(v_pool[:, pg, :, :n], gd.v_cache[:, b, :, p0:p0 + n])
        draft_p = torch.empty_like(draft_c)
        logits_p = torch.empty_like(logits_c)
        dfl.dflash_draft_block_paged(gd.cfg, gd.w, a, ctx2, max(lens), pages, draft_p, gd.status, gd.ws,
                                     logits=logits_p)
        torch.cuda.synchronize()
        gd.check_status()
        for b in range(B):
            out = want[b][2]
            H.assert_logits_close(logits_p[b], out["logits"], f"paged logits b{b} placement {seed}")
            H.assert_drafts_match(draft_p[b].cpu().numpy(), out["logits"], f"paged draft b{b} placement {seed}")
        assert torch.equal(draft_p, draft_c) and torch.equal(logits_p, logits_c)


def test_a_missing_page_is_a_capacity_error_and_its_rows_are_skipped(dfl):
    wl = SMALL
    lens = [300, 45, 0]
    cap = 512
    gd = H.GpuDrafter(dfl, wl, max_rows=max(sum(lens), 16), ctx_capacity=cap)
    h_pad = fused_context(gd, lens)
    # sequence 0 has no page for positions 256..383
    pages, table, k_pool, _ = page_view(dfl, wl, cap // PAGE, 3 * cap // PAGE + 5, 7, holes=[(0, 2)])
    ctx2 = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    n_new = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    dfl.dflash_kv_inject_paged(gd.cfg, gd.w, h_pad, n_new, ctx2, pages, gd.status, gd.ws)
    torch.cuda.synchronize()
    assert int(gd.status.item()) == dfl.ERR_CAPACITY
    # the rows with pages were written
    assert float(k_pool[:, int(table[0, 0])].abs().sum()) > 0.0
