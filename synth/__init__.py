"""Seeded synthetic inputs for the DFlash drafting step.

This module holds workload shapes and random-number recipes only -- none of
the drafting arithmetic. It is the one module that both the CUDA path's
callers (tests, bench, smoke) and the CPU oracle's callers draw inputs from.

Recipes (the pages measure on public suites with trained checkpoints that
are not available here; these shapes and distributions stand in for them):
  weights      N(0, 1/fan_in), rounded to the model dtype
  embedding    N(0, 1)   (a lookup has fan_in = 1)
  norm gains   1 + 0.1 * N(0, 1)
  taps         N(0, 1)   (tapped target hidden states)
  logits       N(0, 1)   (synthetic target logits)
Each tensor has its own generator stream keyed by (seed, tag), so adding a
tensor never shifts the values of another.
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One drafter shape plus the batch / context sizes it is exercised at."""
    name: str
    n_layers: int
    d_target: int
    n_taps: int
    d_model: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ffn: int
    vocab: int
    gamma: int
    dtype: str            # "f32" or "bf16"
    batch: int
    ctx: int              # context length N (or the upper bound when ragged)
    ctx_min: int = -1     # >= 0: ragged lengths drawn from U{ctx_min..ctx}
    cycles: int = 0       # > 0: a draft-verify loop of this many cycles
    seed: int = 0
    rope_theta: float = 1.0e6
    rms_eps: float = 1.0e-6

    @property
    def rows(self) -> int:
        return self.gamma + 1

    @property
    def mask_token_id(self) -> int:
        return self.vocab - 1

    def capacity(self) -> int:
        """KV rows per sequence: context, loop growth, the draft block's R rows."""
        grow = self.cycles * self.rows
        cap = self.ctx + grow + self.rows
        return (cap + 63) // 64 * 64

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


_QWEN3_8B = dict(d_target=4096, n_taps=5, d_model=4096, n_q_heads=32,
                 n_kv_heads=8, head_dim=128, d_ffn=12288, vocab=151936,
                 gamma=16, dtype="bf16")

WORKLOADS = {
    # tiny fp32 drafter, one layer, context 128
    "tiny_f32_L1_N128": Workload(
        "tiny_f32_L1_N128", n_layers=1, d_target=256, n_taps=5, d_model=256,
        n_q_heads=4, n_kv_heads=4, head_dim=64, d_ffn=512, vocab=1024,
        gamma=16, dtype="f32", batch=1, ctx=128, seed=1001),
    # Qwen3-8B-shaped 5-layer bf16 drafter, context 2048, batch 1
    "qwen3_8b_L5_N2048_B1": Workload(
        "qwen3_8b_L5_N2048_B1", n_layers=5, batch=1, ctx=2048, seed=1002,
        **_QWEN3_8B),
    # same drafter, long injected context 32768
    "qwen3_8b_L5_N32768_B1": Workload(
        "qwen3_8b_L5_N32768_B1", n_layers=5, batch=1, ctx=32768, seed=1003,
        **_QWEN3_8B),
    # batched serving: 16 sequences, ragged contexts U{512..8192}
    "qwen3_8b_L5_ragged_B16": Workload(
        "qwen3_8b_L5_ragged_B16", n_layers=5, batch=16, ctx=8192, ctx_min=512,
        seed=1004, **_QWEN3_8B),
    # one-layer version of the same shapes: small enough (~3 GB on the device)
    # for kernel-level profiler captures
    "qwen3_8b_L1_N2048_B1": Workload(
        "qwen3_8b_L1_N2048_B1", n_layers=1, batch=1, ctx=2048, seed=1006, **_QWEN3_8B),
    # one-layer version of the long-context case, for captures of the
    # split-KV attention over 32K keys
    "qwen3_8b_L1_N32768_B1": Workload(
        "qwen3_8b_L1_N32768_B1", n_layers=1, batch=1, ctx=32768, seed=1007, **_QWEN3_8B),
    # one-layer version of the ragged batch-16 case, for kernel-level profiler
    # captures of the batched projections
    "qwen3_8b_L1_ragged_B16": Workload(
        "qwen3_8b_L1_ragged_B16", n_layers=1, batch=16, ctx=8192, ctx_min=512,
        seed=1004, **_QWEN3_8B),
    # full draft-verify loop: 8 layers, batch 4, context 4096, 256 cycles
    "qwen3_8b_L8_loop_B4": Workload(
        "qwen3_8b_L8_loop_B4", n_layers=8, batch=4, ctx=4096, cycles=256,
        seed=1005, **_QWEN3_8B),
}


def tag_seed(seed: int, tag: str) -> int:
    """Independent 63-bit stream key for one named tensor of one workload."""
    return (seed * 0x9E3779B1 + zlib.crc32(tag.encode())) & ((1 << 63) - 1)


def _gen(device, seed: int, tag: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(tag_seed(seed, tag))
    return g


def torch_dtype(name: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def normal(shape, seed: int, tag: str, device="cpu", scale: float = 1.0,
           shift: float = 0.0, dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """shift + scale * N(0,1) of `shape`, drawn in fp32 then cast to dtype."""
    out = torch.randn(tuple(shape), generator=_gen(device, seed, tag),
                      device=device, dtype=torch.float32)
    if scale != 1.0:
        out.mul_(scale)
    if shift != 0.0:
        out.add_(shift)
    return out.to(dtype)


def weights(wl: Workload, device="cpu") -> dict:
    """Drafter parameters of `wl`, stacked over layers, in wl.dtype."""
    dt = torch_dtype(wl.dtype)
    L, D, Dt, T5 = wl.n_layers, wl.d_model, wl.d_target, wl.n_taps
    Hq, Hkv, Dh, F, V = (wl.n_q_heads, wl.n_kv_heads, wl.head_dim, wl.d_ffn,
                         wl.vocab)
    s = wl.seed
    nqkv = (Hq + 2 * Hkv) * Dh

    def lin(shape, tag):
        return normal(shape, s, tag, device, scale=shape[-1] ** -0.5, dtype=dt)

    def gain(shape, tag):
        return normal(shape, s, tag, device, scale=0.1, shift=1.0, dtype=dt)

    return {
        "w_c": lin((D, T5 * Dt), "w_c"),
        "g_c": gain((D,), "g_c"),
        "embed": normal((V, D), s, "embed", device, dtype=dt),
        "g_final": gain((D,), "g_final"),
        "lm_head": lin((V, D), "lm_head"),
        "g_attn": gain((L, D), "g_attn"),
        "w_qkv": lin((L, nqkv, D), "w_qkv"),
        "w_o": lin((L, D, Hq * Dh), "w_o"),
        "g_ffn": gain((L, D), "g_ffn"),
        "w_gateup": lin((L, 2 * F, D), "w_gateup"),
        "w_down": lin((L, D, F), "w_down"),
    }


def taps(wl: Workload, rows: int, tag: str, device="cpu") -> torch.Tensor:
    """[rows, n_taps * Dt] tapped target hidden states, N(0,1), wl.dtype."""
    return normal((rows, wl.n_taps * wl.d_target), wl.seed, "taps/" + tag,
                  device, dtype=torch_dtype(wl.dtype))


def hidden(wl: Workload, rows: int, tag: str, device="cpu") -> torch.Tensor:
    """[rows, D] N(0,1) rows standing in for a fused context feature."""
    return normal((rows, wl.d_model), wl.seed, "hidden/" + tag, device,
                  dtype=torch_dtype(wl.dtype))


def kv_rows(wl: Workload, n: int, tag: str, device="cpu") -> torch.Tensor:
    """[L, B, Hkv, n, Dh] N(0,1) K or V rows for a directly filled cache."""
    shape = (wl.n_layers, wl.batch, wl.n_kv_heads, n, wl.head_dim)
    return normal(shape, wl.seed, "kv/" + tag, device,
                  dtype=torch_dtype(wl.dtype))


def target_logits(wl: Workload, tag: str, device="cpu",
                  dtype=torch.float32) -> torch.Tensor:
    """[B, R, V] N(0,1) synthetic target logits."""
    return normal((wl.batch, wl.rows, wl.vocab), wl.seed, "logits/" + tag,
                  device, dtype=dtype)


def anchors(wl: Workload, tag: str = "anchor") -> np.ndarray:
    """[B] int32 anchor ids drawn uniformly from [0, V-1) (never the mask id)."""
    rng = np.random.default_rng(tag_seed(wl.seed, tag))
    return rng.integers(0, wl.vocab - 1, size=wl.batch, dtype=np.int64).astype(np.int32)


def ctx_lengths(wl: Workload) -> np.ndarray:
    """[B] int32 context lengths: wl.ctx each, or U{ctx_min..ctx} when ragged."""
    if wl.ctx_min < 0:
        return np.full(wl.batch, wl.ctx, dtype=np.int32)
    rng = np.random.default_rng(tag_seed(wl.seed, "ctx_len"))
    return rng.integers(wl.ctx_min, wl.ctx + 1, size=wl.batch,
                        dtype=np.int64).astype(np.int32)


# ---------------------------------------------------------------------------
# Counter-based draws for the draft-verify loop workload. splitmix64
# (S. Vigna, public domain) keyed by (seed, cycle, b, j) gives identical
# integers on every machine, so both sides of a comparison see the same
# acceptance pattern whatever device their noise comes from.
# ---------------------------------------------------------------------------
_M64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _M64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


P_AGREE_16 = 52429   # agreement threshold on a 16-bit hash: 52429 / 65536 = 0.8


def loop_plan(wl: Workload, cycle: int):
    """Per (b, j) of one loop cycle: a 16-bit key and an offset in [1, V-1].
    The synthetic target agrees with draft token j when
    (draft_j * 40503 + key) mod 2^16 < P_AGREE_16 (probability 0.8 over the
    key for every token value, never for the bonus row j = gamma), so whether
    it agrees depends on the drafted token itself; where it does not agree it
    picks (draft_j + offset) mod V, a different token.
    Returns (key16 [B, R] int64, offset [B, R] int64)."""
    B, R, V = wl.batch, wl.rows, wl.vocab
    key16 = np.zeros((B, R), dtype=np.int64)
    offset = np.zeros((B, R), dtype=np.int64)
    for b in range(B):
        for j in range(R):
            key = splitmix64(((wl.seed * 1000003 + cycle) * 4099 + b) * 131 + j)
            key16[b, j] = key >> 48
            offset[b, j] = 1 + (splitmix64(key) % (V - 1))
    return key16, offset


def loop_intended(wl: Workload, key16: torch.Tensor, offset: torch.Tensor,
                  draft: torch.Tensor) -> torch.Tensor:
    """[n, R] int64 tokens the synthetic target makes its argmax, for drafts
    [n, gamma] (any device; integer arithmetic only, so every device gives
    the same tokens). key16 / offset: [n, R] int64 from loop_plan."""
    n, R = draft.shape[0], wl.rows
    base = torch.zeros((n, R), dtype=torch.int64, device=draft.device)
    base[:, : R - 1] = draft.to(torch.int64)
    agree = ((base * 40503 + key16) & 0xFFFF) < P_AGREE_16
    agree[:, R - 1] = False
    return torch.where(agree, base, (base + offset) % wl.vocab)


def loop_target_logits(wl: Workload, cycle: int, draft: torch.Tensor, seqs=None,
                       dtype=torch.float32) -> torch.Tensor:
    """[len(seqs), R, V] synthetic target logits for one loop cycle (all B
    sequences when seqs is None; draft holds the drafts of those sequences).

    N(0,1) noise, then the token loop_intended picks for row j gets
    max(row) + 1, so it is the unique argmax. Uses only integer arithmetic,
    indexing and one max per row, on draft's device."""
    dev = draft.device
    B = wl.batch
    seqs = list(range(B)) if seqs is None else list(seqs)
    noise = normal((B, wl.rows, wl.vocab), wl.seed, f"loop_noise/{cycle}", dev)[seqs]
    key16, offset = loop_plan(wl, cycle)
    intended = loop_intended(wl, torch.as_tensor(key16[seqs], device=dev),
                             torch.as_tensor(offset[seqs], device=dev), draft)
    top = noise.max(dim=-1, keepdim=True).values + 1.0
    noise.scatter_(-1, intended.unsqueeze(-1), top)
    return noise.to(dtype)
