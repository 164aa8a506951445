"""Python binding of libdflash, the GB300 (sm_103a) DFlash drafting step.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels, reached through its C ABI (include/dflash.h). PyTorch provides the
device memory and streams. Functions keep the C names:
dflash_ctx_fuse, dflash_kv_inject, dflash_draft_block, dflash_verify_accept,
plus the sizing / helper calls of the header. There is no CPU fallback: if
the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import _build

F32, BF16 = 0, 1
(OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_DTYPE, ERR_CAPACITY, ERR_ARCH, ERR_CUDA, ERR_TIMEOUT,
 ERR_WORKSPACE, ERR_ALIGN, ERR_TOO_LARGE) = 0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10
K_GEMM, K_ATTN, K_NORM, K_ARGMAX, K_VERIFY = range(5)


class DFlashError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "n_layers", "d_target", "n_taps", "d_model", "n_q_heads", "n_kv_heads", "head_dim",
        "d_ffn", "vocab", "gamma", "mask_token_id", "max_batch", "ctx_capacity")] + [
        ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("dtype", ctypes.c_int)]


class WeightsStruct(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_c", "g_c", "embed", "g_final", "lm_head", "g_attn", "w_qkv", "w_o", "g_ffn",
        "w_gateup", "w_down", "rope_cos", "rope_sin")] + [("rope_positions", ctypes.c_int)]


class Trace(ctypes.Structure):
    _fields_ = [("events", ctypes.POINTER(ctypes.c_void_p)), ("capacity", ctypes.c_int),
                ("count", ctypes.c_int), ("kinds", ctypes.POINTER(ctypes.c_int)),
                ("bytes", ctypes.POINTER(ctypes.c_double)),
                ("flops", ctypes.POINTER(ctypes.c_double))]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
PAGE_KEYS = 128


class KvPages(ctypes.Structure):
    """dflash_kv_pages: page pools [L, n_pages, Hkv, 128, Dh] and a device page
    table [max_batch, pages_per_seq] (tensors kept alive by the object)."""
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("n_pages", ctypes.c_int),
                ("pages_per_seq", ctypes.c_int)]

    def __init__(self, k_pool, v_pool, page_table):
        super().__init__(k_pool.data_ptr(), v_pool.data_ptr(), page_table.data_ptr(), k_pool.shape[1],
                         page_table.shape[1])
        self._keep = (k_pool, v_pool, page_table)


_SIGS = {
    "dflash_abi_version": (_I, []),
    "dflash_status_string": (ctypes.c_char_p, [_I]),
    "dflash_check_config": (_I, [ctypes.POINTER(Config)]),
    "dflash_param_bytes": (_SZ, [ctypes.POINTER(Config), _I]),
    "dflash_kv_cache_bytes": (_SZ, [ctypes.POINTER(Config)]),
    "dflash_workspace_bytes": (_SZ, [ctypes.POINTER(Config), _I]),
    "dflash_workspace_init": (_I, [_P, _SZ, _P]),
    "dflash_ctx_fuse": (_I, [ctypes.POINTER(Config), ctypes.POINTER(WeightsStruct), _P, _I, _P,
                             _P, _SZ, ctypes.POINTER(Trace), _P]),
    "dflash_kv_inject": (_I, [ctypes.POINTER(Config), ctypes.POINTER(WeightsStruct), _P, _P, _I,
                              _I, _P, _P, _P, _P, _P, _SZ, ctypes.POINTER(Trace), _P]),
    "dflash_draft_block": (_I, [ctypes.POINTER(Config), ctypes.POINTER(WeightsStruct), _P, _P,
                                _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                ctypes.POINTER(Trace), _P]),
    "dflash_verify_accept": (_I, [ctypes.POINTER(Config), _P, _I, _P, _I, _P, _P, _P, _P, _SZ,
                                  ctypes.POINTER(Trace), _P]),
    "dflash_rope_tables": (_I, [ctypes.POINTER(Config), _I, _P, _P]),
    "dflash_linear": (_I, [_I, _P, _P, _P, _I, _I, _I, _P, _SZ, _P]),
    "dflash_verify_accept_noalloc": (_I, [ctypes.POINTER(Config), _P, _I, _P, _I, _P, _P, _P, _P]),
    "dflash_selftest_wait_timeout": (_I, [_P, _P]),
    "dflash_attention": (_I, [ctypes.POINTER(Config), _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ,
                              ctypes.POINTER(Trace), _P]),
    "dflash_draft_block_dyn": (_I, [ctypes.POINTER(Config), ctypes.POINTER(WeightsStruct), _P, _P, _P,
                                    _I, _I, _P, _P, _P, _P, _P, _P, _SZ, ctypes.POINTER(Trace), _P]),
    "dflash_verify_accept_dyn": (_I, [ctypes.POINTER(Config), _P, _I, _P, _P, _I, _P, _P, _P, _P, _SZ,
                                      ctypes.POINTER(Trace), _P]),
    "dflash_draft_block_ids": (_I, [ctypes.POINTER(Config), ctypes.POINTER(WeightsStruct), _P, _P, _I, _I,
                                    _P, _P, _P, _P, _P, _P, _SZ, ctypes.POINTER(Trace), _P]),
    "dflash_unmask_step": (_I, [ctypes.POINTER(Config), _P, _P, _P, _I, _I, _P, _SZ, ctypes.POINTER(Trace),
                                _P]),
    "dflash_draft_block_iter": (_I, [ctypes.POINTER(Config), ctypes.POINTER(WeightsStruct), _P, _P, _I, _I,
                                     _P, _P, _I, _P, _P, _P, _P, _P, _SZ, ctypes.POINTER(Trace), _P]),
    "dflash_kv_inject_paged": (_I, [ctypes.POINTER(Config), ctypes.POINTER(WeightsStruct), _P, _P, _I, _I, _P,
                                    ctypes.POINTER(KvPages), _P, _P, _SZ, ctypes.POINTER(Trace), _P]),
    "dflash_draft_block_paged": (_I, [ctypes.POINTER(Config), ctypes.POINTER(WeightsStruct), _P, _P, _I, _I,
                                      ctypes.POINTER(KvPages), _P, _P, _P, _P, _SZ, ctypes.POINTER(Trace), _P]),
    "dflash_draft_block_sample": (_I, [ctypes.POINTER(Config), ctypes.POINTER(WeightsStruct), _P, _P,
                                       _I, _I, _P, _P, ctypes.c_float, ctypes.c_uint64, _P, _P, _P,
                                       _P, _SZ, ctypes.POINTER(Trace), _P]),
    "dflash_verify_sample": (_I, [ctypes.POINTER(Config), _P, _I, _P, _P, _I, ctypes.c_float,
                                  ctypes.c_uint64, _P, _P, _P, _P, _SZ, ctypes.POINTER(Trace), _P]),
}

_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build: bool = True) -> ctypes.CDLL:
    """Loads libdflash.so (building it first when asked and out of date)."""
    global _lib
    if _lib is None:
        if build:
            _build.build_library()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libdflash.so is not built ({_build.LIB}); run __graft_entry__.build()")
        lib = ctypes.CDLL(_build.LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def header_functions() -> list[str]:
    """Names of the functions declared in include/dflash.h."""
    path = os.path.join(_build.INCLUDE, "dflash.h")
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z_0-9]+)\s*\(", text)))


def status_string(s: int) -> str:
    return load().dflash_status_string(s).decode()


def _check(fn: str, s: int):
    if s != OK:
        raise DFlashError(fn, s)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def make_config(n_layers, d_target, n_taps, d_model, n_q_heads, n_kv_heads, head_dim, d_ffn,
                vocab, gamma, mask_token_id, max_batch, ctx_capacity, rms_eps=1e-6,
                rope_theta=1e6, dtype=BF16) -> Config:
    return Config(n_layers, d_target, n_taps, d_model, n_q_heads, n_kv_heads, head_dim, d_ffn,
                  vocab, gamma, mask_token_id, max_batch, ctx_capacity, rms_eps, rope_theta, dtype)


def config_from_workload(wl, max_batch=None, ctx_capacity=None) -> Config:
    return make_config(wl.n_layers, wl.d_target, wl.n_taps, wl.d_model, wl.n_q_heads,
                       wl.n_kv_heads, wl.head_dim, wl.d_ffn, wl.vocab, wl.gamma,
                       wl.mask_token_id, max_batch or wl.batch, ctx_capacity or wl.capacity(),
                       wl.rms_eps, wl.rope_theta, BF16 if wl.dtype == "bf16" else F32)


def dflash_check_config(cfg: Config) -> int:
    return load().dflash_check_config(ctypes.byref(cfg))


def dflash_param_bytes(cfg: Config, kind: int) -> int:
    return load().dflash_param_bytes(ctypes.byref(cfg), kind)


def dflash_kv_cache_bytes(cfg: Config) -> int:
    return load().dflash_kv_cache_bytes(ctypes.byref(cfg))


def dflash_workspace_bytes(cfg: Config, max_rows: int) -> int:
    return load().dflash_workspace_bytes(ctypes.byref(cfg), max_rows)


def dflash_rope_tables(cfg: Config, n_pos: int):
    """(cos, sin) fp32 CPU tensors [n_pos, Dh/2] computed by the library in fp64."""
    half = cfg.head_dim // 2
    c = torch.empty((n_pos, half), dtype=torch.float32)
    s = torch.empty((n_pos, half), dtype=torch.float32)
    _check("dflash_rope_tables", load().dflash_rope_tables(ctypes.byref(cfg), n_pos, c.data_ptr(), s.data_ptr()))
    return c, s


class Weights:
    """Device-resident drafter parameters plus the RoPE tables, and the
    dflash_weights struct that points at them."""

    def __init__(self, cfg: Config, tensors: dict, device="cuda"):
        self.cfg = cfg
        self.t = {k: v.to(device).contiguous() for k, v in tensors.items()}
        self.rope_cos = self.rope_sin = None
        n_rope = 0
        if cfg.rope_theta > 0:
            n_rope = cfg.ctx_capacity
            c, s = dflash_rope_tables(cfg, n_rope)
            self.rope_cos, self.rope_sin = c.to(device), s.to(device)
        t = self.t
        self.struct = WeightsStruct(
            _ptr(t["w_c"]), _ptr(t["g_c"]), _ptr(t["embed"]), _ptr(t["g_final"]),
            _ptr(t["lm_head"]), _ptr(t["g_attn"]), _ptr(t["w_qkv"]), _ptr(t["w_o"]),
            _ptr(t["g_ffn"]), _ptr(t["w_gateup"]), _ptr(t["w_down"]), _ptr(self.rope_cos),
            _ptr(self.rope_sin), n_rope)


class Workspace:
    """Caller-owned scratch buffer sized by dflash_workspace_bytes, zeroed once."""

    def __init__(self, cfg: Config, max_rows: int, device="cuda", stream=None):
        n = dflash_workspace_bytes(cfg, max_rows)
        if n == 0:
            raise DFlashError("dflash_workspace_bytes", dflash_check_config(cfg))
        self.buf = torch.empty(n, dtype=torch.uint8, device=device)
        self.nbytes = n
        _check("dflash_workspace_init",
               load().dflash_workspace_init(self.buf.data_ptr(), n, _stream(stream)))

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


def _tr(trace):
    return ctypes.byref(trace) if trace is not None else None


def dflash_ctx_fuse(cfg, w: Weights, taps, h_ctx, ws: Workspace, trace=None, stream=None):
    T = taps.shape[0] if taps is not None else 0
    _check("dflash_ctx_fuse", load().dflash_ctx_fuse(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(taps), T, _ptr(h_ctx), ws.ptr, ws.nbytes,
        _tr(trace), _stream(stream)))


def dflash_kv_inject(cfg, w: Weights, h_ctx, n_new, ctx_len, k_cache, v_cache, dev_status,
                     ws: Workspace, trace=None, stream=None):
    B, Tmax = h_ctx.shape[0], h_ctx.shape[1]
    _check("dflash_kv_inject", load().dflash_kv_inject(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(h_ctx), _ptr(n_new), B, Tmax,
        _ptr(ctx_len), _ptr(k_cache), _ptr(v_cache), _ptr(dev_status), ws.ptr, ws.nbytes,
        _tr(trace), _stream(stream)))


def dflash_draft_block(cfg, w: Weights, anchor, ctx_len, max_ctx_hint, k_cache, v_cache, draft,
                       dev_status, ws: Workspace, logits=None, layer_dump=None, trace=None,
                       stream=None):
    B = anchor.shape[0]
    _check("dflash_draft_block", load().dflash_draft_block(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(anchor), _ptr(ctx_len), B,
        int(max_ctx_hint), _ptr(k_cache), _ptr(v_cache), _ptr(draft), _ptr(logits),
        _ptr(layer_dump), _ptr(dev_status), ws.ptr, ws.nbytes,
        ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_verify_accept(cfg, target_logits, draft, tau, committed, next_anchor, ws: Workspace,
                         trace=None, stream=None):
    dt = BF16 if target_logits.dtype == torch.bfloat16 else F32
    B = target_logits.shape[0]
    _check("dflash_verify_accept", load().dflash_verify_accept(
        ctypes.byref(cfg), _ptr(target_logits), dt, _ptr(draft), B, _ptr(tau), _ptr(committed),
        _ptr(next_anchor), ws.ptr, ws.nbytes,
        ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_kv_inject_paged(cfg, w: Weights, h_ctx, n_new, ctx_len, pages: KvPages, dev_status, ws: Workspace,
                           trace=None, stream=None):
    B, Tmax = h_ctx.shape[0], h_ctx.shape[1]
    _check("dflash_kv_inject_paged", load().dflash_kv_inject_paged(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(h_ctx), _ptr(n_new), B, Tmax, _ptr(ctx_len),
        ctypes.byref(pages), _ptr(dev_status), ws.ptr, ws.nbytes,
        ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_draft_block_paged(cfg, w: Weights, anchor, ctx_len, max_ctx_hint, pages: KvPages, draft, dev_status,
                             ws: Workspace, logits=None, trace=None, stream=None):
    B = anchor.shape[0]
    _check("dflash_draft_block_paged", load().dflash_draft_block_paged(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(anchor), _ptr(ctx_len), B, int(max_ctx_hint),
        ctypes.byref(pages), _ptr(draft), _ptr(logits), _ptr(dev_status), ws.ptr, ws.nbytes,
        ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_draft_block_dyn(cfg, w: Weights, anchor, ctx_len, gamma_b, max_ctx_hint, k_cache, v_cache,
                           draft, dev_status, ws: Workspace, logits=None, trace=None, stream=None):
    """Drafting pass with block size gamma_b[b] per sequence (draft[b, j] = -1
    for j >= gamma_b[b])."""
    B = anchor.shape[0]
    _check("dflash_draft_block_dyn", load().dflash_draft_block_dyn(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(anchor), _ptr(ctx_len), _ptr(gamma_b), B,
        int(max_ctx_hint), _ptr(k_cache), _ptr(v_cache), _ptr(draft), _ptr(logits), _ptr(dev_status),
        ws.ptr, ws.nbytes, ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_verify_accept_dyn(cfg, target_logits, draft, gamma_b, tau, committed, next_anchor,
                             ws: Workspace, trace=None, stream=None):
    dt = BF16 if target_logits.dtype == torch.bfloat16 else F32
    B = target_logits.shape[0]
    _check("dflash_verify_accept_dyn", load().dflash_verify_accept_dyn(
        ctypes.byref(cfg), _ptr(target_logits), dt, _ptr(draft), _ptr(gamma_b), B, _ptr(tau),
        _ptr(committed), _ptr(next_anchor), ws.ptr, ws.nbytes,
        ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_draft_block_ids(cfg, w: Weights, ids, ctx_len, max_ctx_hint, k_cache, v_cache, draft, dev_status,
                           ws: Workspace, logits=None, trace=None, stream=None):
    """Drafting pass on explicit block inputs ids [B, R]."""
    B = ids.shape[0]
    _check("dflash_draft_block_ids", load().dflash_draft_block_ids(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(ids), _ptr(ctx_len), B, int(max_ctx_hint),
        _ptr(k_cache), _ptr(v_cache), _ptr(draft), _ptr(logits), _ptr(dev_status), ws.ptr, ws.nbytes,
        ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_unmask_step(cfg, logits, draft, ids, steps_left, ws: Workspace, trace=None, stream=None):
    _check("dflash_unmask_step", load().dflash_unmask_step(
        ctypes.byref(cfg), _ptr(logits), _ptr(draft), _ptr(ids), ids.shape[0], int(steps_left), ws.ptr,
        ws.nbytes, ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_draft_block_iter(cfg, w: Weights, anchor, ctx_len, max_ctx_hint, k_cache, v_cache, n_steps, ids,
                            draft, logits, dev_status, ws: Workspace, trace=None, stream=None):
    """n_steps passes of multi-step confidence unmasking."""
    B = anchor.shape[0]
    _check("dflash_draft_block_iter", load().dflash_draft_block_iter(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(anchor), _ptr(ctx_len), B, int(max_ctx_hint),
        _ptr(k_cache), _ptr(v_cache), int(n_steps), _ptr(ids), _ptr(draft), _ptr(logits), _ptr(dev_status),
        ws.ptr, ws.nbytes, ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_draft_block_sample(cfg, w: Weights, anchor, ctx_len, max_ctx_hint, k_cache, v_cache,
                              temperature, seed, draft, logits, dev_status, ws: Workspace, trace=None,
                              stream=None):
    """Sampling drafting pass: draft j ~ softmax(logits_j / temperature);
    logits [B, gamma, V] fp32 receives the raw logits (the verifier's q)."""
    B = anchor.shape[0]
    _check("dflash_draft_block_sample", load().dflash_draft_block_sample(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(anchor), _ptr(ctx_len), B,
        int(max_ctx_hint), _ptr(k_cache), _ptr(v_cache), float(temperature), int(seed) & (2**64 - 1),
        _ptr(draft), _ptr(logits), _ptr(dev_status), ws.ptr, ws.nbytes,
        ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_verify_sample(cfg, target_logits, draft_logits, draft, temperature, seed, tau, committed,
                         next_anchor, ws: Workspace, trace=None, stream=None):
    """Rejection-acceptance verification at temperature > 0."""
    dt = BF16 if target_logits.dtype == torch.bfloat16 else F32
    B = target_logits.shape[0]
    _check("dflash_verify_sample", load().dflash_verify_sample(
        ctypes.byref(cfg), _ptr(target_logits), dt, _ptr(draft_logits), _ptr(draft), B,
        float(temperature), int(seed) & (2**64 - 1), _ptr(tau), _ptr(committed), _ptr(next_anchor),
        ws.ptr, ws.nbytes, ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_verify_accept_noalloc(cfg, target_logits, draft, tau, committed, next_anchor,
                                 stream=None):
    """dflash_verify_accept with its scratch in the library's own device memory
    (no workspace): for callers that cannot allocate device memory."""
    dt = BF16 if target_logits.dtype == torch.bfloat16 else F32
    B = target_logits.shape[0]
    _check("dflash_verify_accept_noalloc", load().dflash_verify_accept_noalloc(
        ctypes.byref(cfg), _ptr(target_logits), dt, _ptr(draft), B, _ptr(tau), _ptr(committed),
        _ptr(next_anchor), _stream(stream)))


def dflash_attention(cfg, q, ctx_len, max_ctx_hint, layer, k_cache, v_cache, out, dev_status,
                     ws: Workspace, trace=None, stream=None):
    """One layer's context attention (the drafting pass's attention step):
    q, out [B*R, Hq*Dh]; the block's K/V already in cache rows ctx_len.."""
    B = ctx_len.shape[0]
    _check("dflash_attention", load().dflash_attention(
        ctypes.byref(cfg), _ptr(q), _ptr(ctx_len), B, int(max_ctx_hint), int(layer), _ptr(k_cache),
        _ptr(v_cache), _ptr(out), _ptr(dev_status), ws.ptr, ws.nbytes,
        ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def dflash_selftest_wait_timeout(dev_status, stream=None):
    """Launches the bounded-wait self-test: dev_status reads ERR_TIMEOUT after ~1 s."""
    _check("dflash_selftest_wait_timeout", load().dflash_selftest_wait_timeout(_ptr(dev_status), _stream(stream)))


def dflash_linear(x, w, y, ws: Workspace, stream=None):
    dt = BF16 if x.dtype == torch.bfloat16 else F32
    M, K = x.shape
    N = w.shape[0]
    _check("dflash_linear", load().dflash_linear(dt, _ptr(x), _ptr(w), _ptr(y), M, N, K, ws.ptr,
                                                 ws.nbytes, _stream(stream)))


class TraceRecorder:
    """Owns CUDA events and host arrays for a dflash_trace."""

    def __init__(self, capacity: int = 512):
        self.capacity = capacity
        self.ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * capacity)]
        for e in self.ev:      # torch creates the CUDA event on first record
            e.record()
        torch.cuda.synchronize()
        self._events = (ctypes.c_void_p * (2 * capacity))(*[e.cuda_event for e in self.ev])
        self._kinds = (ctypes.c_int * capacity)()
        self._bytes = (ctypes.c_double * capacity)()
        self._flops = (ctypes.c_double * capacity)()
        self.struct = Trace(self._events, capacity, 0, self._kinds, self._bytes, self._flops)

    def reset(self):
        self.struct.count = 0

    def records(self):
        """[(kind, bytes, flops, ms)] of the traced launches (synchronises)."""
        torch.cuda.synchronize()
        out = []
        for i in range(self.struct.count):
            ms = self.ev[2 * i].elapsed_time(self.ev[2 * i + 1])
            out.append((self._kinds[i], self._bytes[i], self._flops[i], ms))
        return out
