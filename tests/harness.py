"""Shared set-up for the GPU parity tests: seeded inputs from `synth`, the
C-ABI path through the binding, the oracle on the same inputs, and the
acceptance criteria (written out here so every test applies the same bar).

Acceptance criteria:
  tau, committed tokens, next anchors   bit-exact
  draft tokens                          equal to the oracle's argmax except
                                        where the oracle's top-2 margin < 1e-2
  activations (H_t, KV rows, residual   max |gpu - oracle| <= 3e-2 * RMS(oracle)
  stream after each layer)
  logits                                RMS(gpu - oracle) <= 5e-2 * RMS(oracle)
"""
from __future__ import annotations

import numpy as np
import torch

import synth
from oracle import dflash_ref as ref

ACT_TOL = 3e-2
LOGIT_TOL = 5e-2
MARGIN = 1e-2


def oracle_cfg(wl: synth.Workload, rope_theta=None) -> ref.Cfg:
    return ref.Cfg(wl.n_layers, wl.d_target, wl.n_taps, wl.d_model, wl.n_q_heads,
                   wl.n_kv_heads, wl.head_dim, wl.d_ffn, wl.vocab, wl.gamma, wl.mask_token_id,
                   wl.rms_eps, wl.rope_theta if rope_theta is None else rope_theta)


def assert_act_close(gpu, want, what, tol=ACT_TOL):
    g = ref.f64(gpu)
    w = np.asarray(want, dtype=np.float64)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    rms = float(np.sqrt(np.mean(w * w)))
    err = float(np.max(np.abs(g - w))) if w.size else 0.0
    assert err <= tol * rms, f"{what}: max abs err {err:.3e} > {tol} * rms {rms:.3e}"
    report(what, "max_abs_err/rms", err / max(rms, 1e-30), tol)
    return err / max(rms, 1e-30)


def assert_logits_close(gpu, want, what="logits", tol=LOGIT_TOL):
    g = ref.f64(gpu)
    w = np.asarray(want, dtype=np.float64)
    rel = float(np.sqrt(np.mean((g - w) ** 2)) / np.sqrt(np.mean(w * w)))
    assert rel <= tol, f"{what}: relative rms err {rel:.3e} > {tol}"
    report(what, "rms_err/rms", rel, tol)
    return rel


def assert_drafts_match(gpu_draft, oracle_logits, what="draft", gpu_logits=None):
    """Bit-exact except at near-ties of the oracle (top-2 margin < 1e-2)."""
    d = np.asarray(gpu_draft).reshape(-1)
    lg = np.asarray(oracle_logits, dtype=np.float64).reshape(d.shape[0], -1)
    want = ref.argmax_lowest(lg)
    top2 = np.sort(lg, axis=-1)[:, -2:]
    margin = top2[:, 1] - top2[:, 0]
    bad = (d != want) & (margin >= MARGIN)
    if bad.any():
        rows = np.nonzero(bad)[0]
        detail = []
        for r in rows[:4]:
            item = (f"row {r}: gpu token {d[r]} oracle {want[r]} margin {margin[r]:.4g} "
                    f"oracle logit of gpu token {lg[r, d[r]]:.5f} vs max {lg[r, want[r]]:.5f}")
            if gpu_logits is not None:
                gl = ref.f64(gpu_logits).reshape(d.shape[0], -1)
                item += f"; gpu logits {gl[r, d[r]]:.5f} / {gl[r, want[r]]:.5f}"
            detail.append(item)
        raise AssertionError(f"{what}: {int(bad.sum())} tokens differ outside near-ties: " + "; ".join(detail))
    n_diff = int((d != want).sum())
    report(what, "tokens_differing_at_near_ties", n_diff, 0)
    return n_diff


def report(what, measure, value, tol):
    """Appends one parity measurement to $DFLASH_PARITY_LOG (if set)."""
    import json
    import os
    path = os.environ.get("DFLASH_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": what, "measure": measure, "value": value, "tol": tol}) + "\n")


class GpuDrafter:
    """Device-side state for one workload: weights, KV caches, workspace."""

    def __init__(self, lib, wl: synth.Workload, max_rows: int = 4096, device="cuda",
                 ctx_capacity=None, weights=None):
        self.lib, self.wl, self.device = lib, wl, device
        self.cfg = lib.config_from_workload(wl, ctx_capacity=ctx_capacity)
        self.W = weights if weights is not None else synth.weights(wl, device)
        self.w = lib.Weights(self.cfg, self.W, device)
        self.ws = lib.Workspace(self.cfg, max_rows, device)
        dt = synth.torch_dtype(wl.dtype)
        shape = (wl.n_layers, self.cfg.max_batch, wl.n_kv_heads, self.cfg.ctx_capacity, wl.head_dim)
        self.k_cache = torch.zeros(shape, dtype=dt, device=device)
        self.v_cache = torch.zeros(shape, dtype=dt, device=device)
        self.ctx_len = torch.zeros(self.cfg.max_batch, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.dt = dt

    def check_status(self):
        s = int(self.status.item())
        assert s == 0, f"device status {s}: {self.lib.status_string(s)}"

    def fuse(self, taps):
        h = torch.empty((taps.shape[0], self.wl.d_model), dtype=self.dt, device=self.device)
        self.lib.dflash_ctx_fuse(self.cfg, self.w, taps, h, self.ws)
        return h

    def inject(self, h_ctx, n_new):
        """h_ctx [B, Tmax, D]; n_new int list/array of length B."""
        nn = torch.as_tensor(np.asarray(n_new, dtype=np.int32), device=self.device)
        self.lib.dflash_kv_inject(self.cfg, self.w, h_ctx, nn, self.ctx_len[: h_ctx.shape[0]],
                                  self.k_cache, self.v_cache, self.status, self.ws)

    def draft(self, anchors, max_ctx, want_logits=False, want_dump=False, trace=None):
        B = len(anchors)
        wl = self.wl
        a = torch.as_tensor(np.asarray(anchors, dtype=np.int32), device=self.device)
        draft = torch.empty((B, wl.gamma), dtype=torch.int32, device=self.device)
        logits = (torch.empty((B, wl.gamma, wl.vocab), dtype=torch.float32, device=self.device)
                  if want_logits else None)
        dump = (torch.empty((wl.n_layers + 1, B * wl.rows, wl.d_model), dtype=torch.float32,
                            device=self.device) if want_dump else None)
        self.lib.dflash_draft_block(self.cfg, self.w, a, self.ctx_len[:B], max_ctx, self.k_cache,
                                    self.v_cache, draft, self.status, self.ws, logits=logits,
                                    layer_dump=dump, trace=trace)
        return draft, logits, dump

    def verify(self, target_logits, draft):
        B = target_logits.shape[0]
        R = self.wl.rows
        tau = torch.empty(B, dtype=torch.int32, device=self.device)
        committed = torch.empty((B, R), dtype=torch.int32, device=self.device)
        nxt = torch.empty(B, dtype=torch.int32, device=self.device)
        self.lib.dflash_verify_accept(self.cfg, target_logits, draft, tau, committed, nxt, self.ws)
        return tau, committed, nxt


def oracle_weights_layer_view(W: dict) -> dict:
    """The oracle accepts the same tensors (it converts to float64 per use)."""
    return W
