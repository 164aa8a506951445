"""GPU: one layer's context attention (dflash_attention, the split-KV tcgen05
kernels of the drafting pass) against the oracle's attention over the
concatenation [K_ctx ; K_block] ("KV Injection 메커니즘" K_i / V_i equations,
bidirectional inside the block): ragged contexts with an empty one, head
dimensions 64 and 128, the cluster merge and the workspace merge of split
partials, and a 32768-key context of the Qwen3-8B-shaped heads."""
import os

import numpy as np
import pytest
import torch

import synth
from oracle import dflash_ref as ref
from tests import harness as H

pytestmark = pytest.mark.gpu

WL64 = synth.Workload("attn_dh64", n_layers=2, d_target=128, n_taps=5, d_model=256,
                      n_q_heads=8, n_kv_heads=2, head_dim=64, d_ffn=384, vocab=1003, gamma=16,
                      dtype="bf16", batch=3, ctx=900, seed=41)
WL128 = WL64.replace(name="attn_dh128", head_dim=128, seed=43)


@pytest.fixture(scope="module")
def dfl(lib):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return lib


def run_attention(dfl, wl, lens, layer, splits=None, capacity=None):
    B, R = wl.batch, wl.rows
    cfg = dfl.config_from_workload(wl, ctx_capacity=capacity)
    ws = dfl.Workspace(cfg, 16)
    n = int(max(lens)) + R
    k = synth.kv_rows(wl, n, "attn/k", "cuda")
    v = synth.kv_rows(wl, n, "attn/v", "cuda")
    shape = (wl.n_layers, B, wl.n_kv_heads, cfg.ctx_capacity, wl.head_dim)
    k_cache = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    v_cache = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    k_cache[:, :, :, :n] = k
    v_cache[:, :, :, :n] = v
    # rows beyond each context + block hold values attention must not read
    for b, nb in enumerate(lens):
        k_cache[:, b, :, nb + R:] = float("nan")
        v_cache[:, b, :, nb + R:] = float("nan")
    q = synth.normal((B * R, wl.n_q_heads * wl.head_dim), wl.seed, "attn/q", "cuda", dtype=torch.bfloat16)
    out = torch.empty_like(q)
    ctx_len = torch.as_tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    old = os.environ.get("DFLASH_ATTN_SPLITS")
    if splits is not None:
        os.environ["DFLASH_ATTN_SPLITS"] = str(splits)
    try:
        dfl.dflash_attention(cfg, q, ctx_len, max(lens), layer, k_cache, v_cache, out, status, ws)
        torch.cuda.synchronize()
    finally:
        if old is None:
            os.environ.pop("DFLASH_ATTN_SPLITS", None)
        else:
            os.environ["DFLASH_ATTN_SPLITS"] = old
    assert int(status.item()) == 0
    oc = H.oracle_cfg(wl)
    for b, nb in enumerate(lens):
        kb = ref.f64(k_cache[layer, b, :, :nb + R])
        vb = ref.f64(v_cache[layer, b, :, :nb + R])
        qb = ref.f64(q[b * R:(b + 1) * R]).reshape(R, wl.n_q_heads, wl.head_dim)
        want = ref.attention(oc, qb, kb, vb).reshape(R, -1)
        H.assert_act_close(out[b * R:(b + 1) * R], want, f"attention b{b} n={nb} layer {layer}")


@pytest.mark.parametrize("wl", [WL64, WL128], ids=["dh64", "dh128"])
@pytest.mark.parametrize("splits", [None, 16], ids=["planned", "workspace_merge"])
def test_attention_matches_the_oracle(dfl, wl, splits):
    run_attention(dfl, wl, [900, 250, 0], layer=1, splits=splits, capacity=1024)


def test_attention_32k_context_matches_the_oracle(dfl):
    wl = synth.WORKLOADS["qwen3_8b_L1_N32768_B1"]
    run_attention(dfl, wl, [wl.ctx], layer=0)
