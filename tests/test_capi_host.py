"""Host-side checks of the C-ABI library: it loads, exports every function
that include/dflash.h declares, and its pure-host calls (config checks,
sizing, RoPE tables, argument validation) behave without a GPU."""
import ctypes
import os

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "memory_table.txt")


def read_golden():
    out = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        key, val, tol = line.split()[:3]
        out[key] = (float(val), float(tol))
    return out


def test_library_exports_every_header_function(lib):
    names = lib.header_functions()
    assert "dflash_draft_block" in names and "dflash_verify_accept" in names
    so = ctypes.CDLL(lib.lib_path())
    missing = [n for n in names if not hasattr(so, n)]
    assert not missing, missing
    assert lib.load().dflash_abi_version() == 1


def test_status_strings(lib):
    for s in range(0, -11, -1):
        assert lib.status_string(s) != "unknown status"
    assert lib.status_string(-99) == "unknown status"


def test_workload_configs_are_accepted(lib):
    for wl in synth.WORKLOADS.values():
        cfg = lib.config_from_workload(wl)
        assert lib.dflash_check_config(cfg) == lib.OK, wl.name
        assert lib.dflash_workspace_bytes(cfg, 4096) > 0


def test_bad_configs_are_rejected(lib):
    wl = synth.WORKLOADS["qwen3_8b_L5_N2048_B1"]
    good = lib.config_from_workload(wl)
    for field, value, want in [("gamma", 0, lib.ERR_INVALID_ARG), ("gamma", 17, lib.ERR_INVALID_ARG),
                               ("head_dim", 96, lib.ERR_SHAPE), ("n_kv_heads", 5, lib.ERR_SHAPE),
                               ("d_model", 4000, lib.ERR_SHAPE), ("dtype", 7, lib.ERR_DTYPE),
                               ("mask_token_id", wl.vocab, lib.ERR_INVALID_ARG),
                               ("ctx_capacity", 10, lib.ERR_INVALID_ARG)]:
        cfg = lib.make_config(*[getattr(good, f) for f, _ in lib.Config._fields_])
        setattr(cfg, field, value)
        assert lib.dflash_check_config(cfg) == want, field


def test_memory_table_of_the_pages(lib):
    """W_c and the fusion's activations for the page's D = 2048 bf16 example."""
    g = read_golden()
    cfg = lib.make_config(5, 2048, 5, 2048, 16, 4, 128, 6144, 32000, 16, 31999, 1, 4096)
    wc = lib.dflash_param_bytes(cfg, 0)
    assert wc == 5 * 2048 * 2048 * 2
    v, tol = g["w_c_param_bytes"]
    assert abs(wc - v) / v <= tol
    seq = 2048
    fin = seq * cfg.n_taps * cfg.d_target * 2
    fout = seq * cfg.d_model * 2
    for key, got in [("fuse_input_activation_bytes", fin), ("fuse_output_activation_bytes", fout)]:
        v, tol = g[key]
        assert abs(got - v) / v <= tol, key
    # decode time: the same projection over one block of 16 rows (in + out)
    blk = 16 * cfg.n_taps * cfg.d_target * 2 + 16 * cfg.d_model * 2
    assert blk < g["decode_block_activation_max"][0]


def test_param_bytes_of_qwen3_8b_shape(lib):
    wl = synth.WORKLOADS["qwen3_8b_L5_N2048_B1"]
    cfg = lib.config_from_workload(wl)
    per_layer = ((32 + 16) * 128 * 4096 + 4096 * 4096 + 2 * 12288 * 4096 + 4096 * 12288 + 2 * 4096) * 2
    assert lib.dflash_param_bytes(cfg, 3) == 5 * per_layer
    assert lib.dflash_param_bytes(cfg, 2) == 151936 * 4096 * 2
    assert lib.dflash_kv_cache_bytes(cfg) == 5 * 1 * 8 * wl.capacity() * 128 * 2


def test_rope_tables_match_closed_form(lib):
    cfg = lib.config_from_workload(synth.WORKLOADS["tiny_f32_L1_N128"])
    c, s = lib.dflash_rope_tables(cfg, 300)
    half = cfg.head_dim // 2
    p = np.arange(300)[:, None]
    j = np.arange(half)[None, :]
    ang = p * cfg.rope_theta ** (-2.0 * j / cfg.head_dim)
    np.testing.assert_allclose(c.numpy(), np.cos(ang), atol=2e-7)
    np.testing.assert_allclose(s.numpy(), np.sin(ang), atol=2e-7)


def test_null_arguments_rejected_before_any_launch(lib):
    L = lib.load()
    cfg = lib.config_from_workload(synth.WORKLOADS["tiny_f32_L1_N128"])
    w = lib.WeightsStruct()
    assert L.dflash_draft_block(ctypes.byref(cfg), ctypes.byref(w), None, None, 1, 0, None, None,
                                None, None, None, None, None, 0, None, None) == lib.ERR_INVALID_ARG
    assert L.dflash_verify_accept(ctypes.byref(cfg), None, 0, None, 1, None, None, None, None, 0,
                                  None, None) == lib.ERR_INVALID_ARG
    assert L.dflash_kv_inject(ctypes.byref(cfg), ctypes.byref(w), None, None, 1, 4, None, None,
                              None, None, None, 0, None, None) == lib.ERR_INVALID_ARG
    # T == 0 and B == 0 are no-ops
    assert L.dflash_ctx_fuse(ctypes.byref(cfg), ctypes.byref(w), None, 0, None, None, 0, None,
                             None) == lib.OK
    assert L.dflash_kv_inject(ctypes.byref(cfg), ctypes.byref(w), None, None, 0, 4, None, None,
                              None, None, None, 0, None, None) == lib.OK
    # batch beyond max_batch
    assert L.dflash_verify_accept(ctypes.byref(cfg), 1, 0, 1, cfg.max_batch + 1, 1, 1, 1, 1, 1,
                                  None, None) == lib.ERR_INVALID_ARG
    assert L.dflash_linear(5, None, None, None, 1, 1, 64, None, 0, None) == lib.ERR_DTYPE


def test_sampling_entry_points_reject_bad_arguments_before_any_launch(lib):
    L = lib.load()
    cfg = lib.config_from_workload(synth.WORKLOADS["tiny_f32_L1_N128"])
    w = lib.WeightsStruct()
    fake = 256  # any non-null address: nothing is dereferenced on the host
    # temperature must be > 0 and finite; the logits buffer is required
    for t in (0.0, -1.0, float("inf"), float("nan")):
        assert L.dflash_draft_block_sample(ctypes.byref(cfg), ctypes.byref(w), fake, fake, 1, 0, fake, fake,
                                           t, 1, fake, fake, fake, fake, 1 << 30, None,
                                           None) == lib.ERR_INVALID_ARG
        assert L.dflash_verify_sample(ctypes.byref(cfg), fake, lib.F32, fake, fake, 1, t, 1, fake, fake,
                                      fake, fake, 1 << 30, None, None) == lib.ERR_INVALID_ARG
    assert L.dflash_draft_block_sample(ctypes.byref(cfg), ctypes.byref(w), fake, fake, 1, 0, fake, fake,
                                       1.0, 1, fake, None, fake, fake, 1 << 30, None,
                                       None) == lib.ERR_INVALID_ARG
    assert L.dflash_verify_sample(ctypes.byref(cfg), fake, lib.F32, None, fake, 1, 1.0, 1, fake, fake, fake,
                                  fake, 1 << 30, None, None) == lib.ERR_INVALID_ARG
    assert L.dflash_verify_sample(ctypes.byref(cfg), fake, 7, fake, fake, 1, 1.0, 1, fake, fake, fake,
                                  fake, 1 << 30, None, None) == lib.ERR_DTYPE
    assert L.dflash_verify_sample(ctypes.byref(cfg), fake, lib.F32, fake, fake, cfg.max_batch + 1, 1.0, 1,
                                  fake, fake, fake, fake, 1 << 30, None, None) == lib.ERR_INVALID_ARG
    # workspace too small
    assert L.dflash_verify_sample(ctypes.byref(cfg), fake, lib.F32, fake, fake, 1, 1.0, 1, fake, fake, fake,
                                  fake, 16, None, None) == lib.ERR_WORKSPACE


def test_per_sequence_gamma_calls_require_the_gamma_array(lib):
    L = lib.load()
    cfg = lib.config_from_workload(synth.WORKLOADS["tiny_f32_L1_N128"])
    w = lib.WeightsStruct()
    fake = 256
    assert L.dflash_draft_block_dyn(ctypes.byref(cfg), ctypes.byref(w), fake, fake, None, 1, 0, fake, fake, fake,
                                    None, fake, fake, 1 << 30, None, None) == lib.ERR_INVALID_ARG
    assert L.dflash_verify_accept_dyn(ctypes.byref(cfg), fake, lib.F32, fake, None, 1, fake, fake, fake, fake,
                                      1 << 30, None, None) == lib.ERR_INVALID_ARG


def test_unmasking_calls_reject_bad_arguments(lib):
    L = lib.load()
    cfg = lib.config_from_workload(synth.WORKLOADS["tiny_f32_L1_N128"])
    w = lib.WeightsStruct()
    fake = 256
    assert L.dflash_unmask_step(ctypes.byref(cfg), fake, fake, fake, 1, 0, fake, 1 << 30, None,
                                None) == lib.ERR_INVALID_ARG          # steps_left >= 1
    assert L.dflash_unmask_step(ctypes.byref(cfg), None, fake, fake, 1, 1, fake, 1 << 30, None,
                                None) == lib.ERR_INVALID_ARG
    assert L.dflash_unmask_step(ctypes.byref(cfg), fake, fake, fake, 1, 1, fake, 16, None,
                                None) == lib.ERR_WORKSPACE
    for n in (0, cfg.gamma + 1):                                      # 1 <= n_steps <= gamma
        assert L.dflash_draft_block_iter(ctypes.byref(cfg), ctypes.byref(w), fake, fake, 1, 0, fake, fake, n,
                                         fake, fake, fake, fake, fake, 1 << 30, None, None) == lib.ERR_INVALID_ARG
    assert L.dflash_draft_block_ids(ctypes.byref(cfg), ctypes.byref(w), None, fake, 1, 0, fake, fake, fake, None,
                                    fake, fake, 1 << 30, None, None) == lib.ERR_INVALID_ARG


def test_paged_calls_reject_missing_or_short_page_views(lib):
    L = lib.load()
    cfg = lib.config_from_workload(synth.WORKLOADS["tiny_f32_L1_N128"])
    w = lib.WeightsStruct()
    fake = 256
    for pages in (None, lib.KvPages.__new__(lib.KvPages)):
        if pages is not None:   # pools and table set, but no pages
            ctypes.Structure.__init__(pages, fake, fake, fake, 0, 1)
        arg = ctypes.byref(pages) if pages is not None else None
        assert L.dflash_draft_block_paged(ctypes.byref(cfg), ctypes.byref(w), fake, fake, 1, 0, arg, fake, None,
                                          fake, fake, 1 << 30, None, None) == lib.ERR_INVALID_ARG
        assert L.dflash_kv_inject_paged(ctypes.byref(cfg), ctypes.byref(w), fake, fake, 1, 4, fake, arg, fake, fake,
                                        1 << 30, None, None) == lib.ERR_INVALID_ARG


def test_drafting_batch_limit_is_the_configured_max_batch(lib):
    """A drafting pass takes any B up to cfg.max_batch, including passes of more
    than 512 block rows (several token tiles); B above max_batch (or below 1)
    is refused before anything else is looked at. With null pointers an
    accepted B proceeds to the pointer checks (ERR_INVALID_ARG as well, so the
    accepted sizes are told apart by a config whose max_batch is smaller)."""
    wl = synth.WORKLOADS["qwen3_8b_L5_N2048_B1"].replace(batch=40)
    w = lib.WeightsStruct()
    L = lib.load()
    small = lib.config_from_workload(wl.replace(batch=30))
    big = lib.config_from_workload(wl)
    assert lib.dflash_check_config(big) == lib.OK
    for cfg, B in [(small, 31), (small, 0), (big, 41)]:
        assert L.dflash_draft_block(ctypes.byref(cfg), ctypes.byref(w), None, None, B, 0, None, None,
                                    None, None, None, None, None, 0, None, None) == lib.ERR_INVALID_ARG
    # 40 sequences of 17 rows (680 > 512) pass the size checks and stop at the
    # first null pointer, which is not a size error
    for B in (30, 31, 40):
        st = L.dflash_draft_block(ctypes.byref(big), ctypes.byref(w), None, None, B, 0, None, None,
                                  None, None, None, None, None, 0, None, None)
        assert st == lib.ERR_INVALID_ARG and st != lib.ERR_TOO_LARGE
