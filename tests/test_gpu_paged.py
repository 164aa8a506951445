"""GPU parity of the paged KV cache: injection and drafting through a page
table must give exactly the contiguous cache's rows, drafts and logits (the
contiguous path is pinned to the oracle elsewhere), wherever the pages sit in
the pool; a missing page is a capacity error."""
import numpy as np
import pytest
import torch

import synth
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


def fused_context(gd, lens):
    wl = gd.wl
    total = int(sum(lens))
    taps = synth.taps(wl, total, "ctx", "cuda")
    h = gd.fuse(taps)
    h_pad = torch.zeros((len(lens), max(lens), wl.d_model), dtype=gd.dt, device="cuda")
    offs = np.concatenate([[0], np.cumsum(lens)])
    for b in range(len(lens)):
        h_pad[b, : lens[b]] = h[offs[b]:offs[b + 1]]
    return h_pad


@pytest.mark.parametrize("wl", [SMALL, synth.WORKLOADS["tiny_f32_L1_N128"].replace(batch=2)],
                         ids=["bf16_tcgen05", "fp32_simt"])
def test_paged_cache_gives_the_contiguous_results_bit_for_bit(dfl, wl):
    lens = [300, 45, 0][: wl.batch] if wl.batch == 3 else [200, 9]
    cap = 512
    gd = H.GpuDrafter(dfl, wl, max_rows=max(sum(lens), 16), ctx_capacity=cap)
    B = wl.batch
    h_pad = fused_context(gd, lens)
    gd.inject(h_pad, lens)
    n_new = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    anchors = synth.anchors(wl)
    a = torch.as_tensor(np.asarray(anchors, dtype=np.int32), device="cuda")
    draft_c, logits_c, _ = gd.draft(anchors, max(lens), want_logits=True)
    torch.cuda.synchronize()
    gd.check_status()
    for seed in (1, 2):   # two different placements of the pages in the pool
        pages, table, k_pool, v_pool = page_view(dfl, wl, cap // PAGE, B * cap // PAGE + 5, seed)
        ctx2 = torch.zeros(B, dtype=torch.int32, device="cuda")
        dfl.dflash_kv_inject_paged(gd.cfg, gd.w, h_pad, n_new, ctx2, pages, gd.status, gd.ws)
        torch.cuda.synchronize()
        gd.check_status()
        assert ctx2.cpu().tolist() == list(lens)
        for b in range(B):
            for p0 in range(0, lens[b], PAGE):
                n = min(PAGE, lens[b] - p0)
                pg = int(table[b, p0 // PAGE])
                assert torch.equal(k_pool[:, pg, :, :n], gd.k_cache[:, b, :, p0:p0 + n])
                assert torch.equal(v_pool[:, pg, :, :n], gd.v_cache[:, b, :, p0:p0 + n])
        draft_p = torch.empty_like(draft_c)
        logits_p = torch.empty_like(logits_c)
        dfl.dflash_draft_block_paged(gd.cfg, gd.w, a, ctx2, max(lens), pages, draft_p, gd.status, gd.ws,
                                     logits=logits_p)
        torch.cuda.synchronize()
        gd.check_status()
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
