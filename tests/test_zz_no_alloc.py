"""The allocation-free verify-accept entry point against the workspace one.

dflash_verify_accept_noalloc exists for callers that cannot allocate device
memory (a serving engine whose pool owns the GPU's memory, a plugin inside
another runtime's step, a hot loop that cannot afford cudaMalloc's implicit
synchronisation). Its scratch lives in a fixed array inside the library, so
this test checks that it gives exactly the results of dflash_verify_accept,
on two calls in a row (the second finds the array as the first left it).
The file sorts last so that a stopped run has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from oracle import dflash_ref as ref

pytestmark = pytest.mark.gpu

WL = synth.Workload("noalloc_verify", n_layers=1, d_target=128, n_taps=5, d_model=256,
                    n_q_heads=8, n_kv_heads=2, head_dim=128, d_ffn=384, vocab=151936, gamma=16,
                    dtype="bf16", batch=6, ctx=64, seed=21)


def planted(wl, seed, dtype):
    logits = synth.target_logits(wl, f"noalloc{seed}", "cuda", torch.float32)
    rng = np.random.default_rng(seed)
    draft = rng.integers(0, wl.vocab, size=(wl.batch, wl.gamma)).astype(np.int32)
    for b in range(wl.batch):
        for j in range([0, wl.gamma, 3, 7, 1, 11][b % 6]):
            logits[b, j, int(draft[b, j])] = logits[b, j].max() + 1.0
    return logits.to(dtype), torch.as_tensor(draft, device="cuda")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_verify_matches_workspace_verify(lib, dtype):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    cfg = lib.config_from_workload(WL)
    ws = lib.Workspace(cfg, 16)
    B, R = WL.batch, WL.rows
    for call in range(2):
        logits, draft = planted(WL, 100 + call, dtype)
        outs = []
        for fn in ("ws", "noalloc"):
            tau = torch.full((B,), -7, dtype=torch.int32, device="cuda")
            committed = torch.full((B, R), -7, dtype=torch.int32, device="cuda")
            nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
            if fn == "ws":
                lib.dflash_verify_accept(cfg, logits, draft, tau, committed, nxt, ws)
            else:
                lib.dflash_verify_accept_noalloc(cfg, logits, draft, tau, committed, nxt)
            torch.cuda.synchronize()
            outs.append((tau.cpu().numpy(), committed.cpu().numpy(), nxt.cpu().numpy()))
        for a, b in zip(outs[0], outs[1]):
            np.testing.assert_array_equal(a, b)   # integer outputs: exact
        assert (outs[1][0] >= 1).all() and (outs[1][0] <= R).all()
        # and both are the oracle's greedy acceptance
        d_np = draft.cpu().numpy()
        for b in range(B):
            t, c, n = ref.verify_accept(logits[b].float().cpu(), d_np[b])
            assert int(outs[1][0][b]) == t and int(outs[1][2][b]) == n
            np.testing.assert_array_equal(outs[1][1][b], c)


def _both(lib, cfg, ws, logits, draft):
    """(tau, committed, next anchor) of the workspace call and of the
    allocation-free call on the same inputs."""
    B, R = logits.shape[0], logits.shape[1]
    outs = []
    for fn in ("ws", "noalloc"):
        tau = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        committed = torch.full((B, R), -7, dtype=torch.int32, device="cuda")
        nxt = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        if fn == "ws":
            lib.dflash_verify_accept(cfg, logits, draft, tau, committed, nxt, ws)
        else:
            lib.dflash_verify_accept_noalloc(cfg, logits, draft, tau, committed, nxt)
        torch.cuda.synchronize()
        outs.append((tau.cpu().numpy(), committed.cpu().numpy(), nxt.cpu().numpy()))
    return outs


def test_noalloc_verify_at_the_array_edge_and_after_larger_calls(lib):
    """963 sequences of 17 rows (16371 of the array's 16384 key slots), then a
    small call, then the full-size call again: every call must match the
    workspace call, whatever an earlier, larger call left in the array."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    wl = WL.replace(vocab=1003, batch=963)
    cfg = lib.config_from_workload(wl)
    ws = lib.Workspace(cfg, 16)
    for call, B in enumerate([963, 5, 963, 1]):
        logits, draft = planted(wl.replace(batch=B), 200 + call, torch.float32)
        outs = _both(lib, cfg, ws, logits, draft)
        for a, b in zip(outs[0], outs[1]):
            np.testing.assert_array_equal(a, b)
        assert (outs[1][0] >= 1).all() and (outs[1][0] <= wl.rows).all()


def test_noalloc_verify_rejects_oversized_batches(lib):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    big = WL.replace(batch=1200)
    cfg = lib.config_from_workload(big)
    L = lib.load()
    one = torch.zeros(1, device="cuda")
    st = L.dflash_verify_accept_noalloc(ctypes.byref(cfg), one.data_ptr(), lib.F32, one.data_ptr(),
                                        1200, one.data_ptr(), one.data_ptr(), one.data_ptr(), None)
    assert st == lib.ERR_TOO_LARGE
