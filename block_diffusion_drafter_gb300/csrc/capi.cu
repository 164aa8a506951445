// C ABI of the drafting step: argument validation, workspace layout, and the
// launch sequences of dflash_ctx_fuse / dflash_kv_inject / dflash_draft_block
// / dflash_verify_accept. Host code only; every step of the path runs in the
// kernels of gemm.cu, attention.cu and small.cu.
#include <cmath>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "internal.h"

using namespace dfl;

namespace {

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline int elem_bytes(const dflash_config* c) { return c->dtype == DFLASH_BF16 ? 2 : 4; }
inline int rows_per_block(const dflash_config* c) { return c->gamma + 1; }

struct WsLayout {
  size_t h, xn, q, attn_o, act, z, ss, lm_keys, v_keys, v_count, samp, attn_part;
  size_t row_ss;
  size_t fixed;  // bytes before row_ss
};

WsLayout ws_layout(const dflash_config* c) {
  WsLayout L{};
  const size_t es = elem_bytes(c);
  const size_t R = rows_per_block(c);
  const size_t rows = static_cast<size_t>(c->max_batch) * R;
  const size_t D = c->d_model, HD = static_cast<size_t>(c->n_q_heads) * c->head_dim;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off = align256(off + bytes); return o; };
  // bf16 models keep the activations that feed a projection as hi + lo bf16
  // halves (two row blocks), fp32 models as one block
  const size_t parts = c->dtype == DFLASH_BF16 ? 2 : 1;
  L.h = take(rows * D * 4);
  L.xn = take(parts * rows * D * es);
  L.q = take(rows * HD * es);
  L.attn_o = take(parts * rows * HD * es);
  L.act = take(parts * rows * static_cast<size_t>(c->d_ffn) * es);
  L.z = take(parts * static_cast<size_t>(c->max_batch) * c->gamma * D * es);
  L.ss = take(rows * (D / kBM) * 4);
  // per (LM-head tile, mask row): the tile's packed argmax key
  L.lm_keys = take(static_cast<size_t>((c->vocab + kBM - 1) / kBM) * c->max_batch * c->gamma * 8);
  L.v_keys = take(rows * 8);
  L.v_count = take(static_cast<size_t>(c->max_batch) * 4);
  L.samp = take(dfl::sample_ws_bytes(c->max_batch, c->gamma, c->vocab));
  // split-KV partials of long contexts (tcgen05 attention, bf16 drafters)
  L.attn_part = take(c->dtype == DFLASH_BF16
                         ? static_cast<size_t>(dfl::kAttnMaxSlots) * dfl::attn_slot_floats(c->head_dim) * 4
                         : 0);
  L.row_ss = off;
  L.fixed = off;
  return L;
}

// Per context row of a fusion call: fp32 u = W_c x (D floats) followed, in a
// second region, by its D/128 partial sums of squares.
size_t row_ss_bytes_per_row(const dflash_config* c) {
  return static_cast<size_t>(c->d_model) * 4 + static_cast<size_t>(c->d_model / kBM) * 4;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

}  // namespace

namespace dfl {
dflash_status check_arch() {
  static int cached[64] = {};  // 0 unknown, 1 ok, 2 bad
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH_ERR_CUDA;
  int& s = cached[dev & 63];
  if (s == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    s = (major == 10 && minor == 3) ? 1 : 2;
  }
  return s == 1 ? DFLASH_OK : DFLASH_ERR_ARCH;
}

bool use_pdl() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("DFLASH_PDL");
    v = (e != nullptr && e[0] == '0') ? 0 : 1;
  }
  return v == 1;
}
}  // namespace dfl

namespace {

// Records trace events around one launch.
struct Tracer {
  dflash_trace* t;
  cudaStream_t s;
  int idx = -1;
  void before(int kind, double bytes, double flops) {
    if (t == nullptr || t->count >= t->capacity) { idx = -1; return; }
    idx = t->count;
    t->kinds[idx] = kind;
    t->bytes[idx] = bytes;
    t->flops[idx] = flops;
    cudaEventRecord(static_cast<cudaEvent_t>(t->events[2 * idx]), s);
  }
  void after() {
    if (idx < 0) return;
    cudaEventRecord(static_cast<cudaEvent_t>(t->events[2 * idx + 1]), s);
    t->count = idx + 1;
    idx = -1;
  }
};

#define DFL_CUDA(call)                          \
  do {                                          \
    if ((call) != cudaSuccess) return DFLASH_ERR_CUDA; \
  } while (0)

}  // namespace

extern "C" {

int dflash_abi_version(void) { return DFLASH_ABI_VERSION; }

const char* dflash_status_string(dflash_status s) {
  switch (s) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_SHAPE: return "unsupported shape";
    case DFLASH_ERR_DTYPE: return "unsupported dtype";
    case DFLASH_ERR_CAPACITY: return "kv cache capacity exceeded";
    case DFLASH_ERR_ARCH: return "device is not sm_103";
    case DFLASH_ERR_CUDA: return "cuda error";
    case DFLASH_ERR_TIMEOUT: return "device wait timed out";
    case DFLASH_ERR_WORKSPACE: return "workspace missing or too small";
    case DFLASH_ERR_ALIGN: return "pointer not 16-byte aligned";
    case DFLASH_ERR_TOO_LARGE: return "request beyond the fixed maximum size";
  }
  return "unknown status";
}

dflash_status dflash_check_config(const dflash_config* c) {
  if (c == nullptr) return DFLASH_ERR_INVALID_ARG;
  if (c->dtype != DFLASH_BF16 && c->dtype != DFLASH_F32) return DFLASH_ERR_DTYPE;
  if (c->n_layers < 1 || c->d_target < 1 || c->n_taps < 1 || c->d_model < 1 || c->n_q_heads < 1 ||
      c->n_kv_heads < 1 || c->d_ffn < 1 || c->vocab < 2 || c->max_batch < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (c->gamma < 1 || c->gamma > DFLASH_MAX_GAMMA) return DFLASH_ERR_INVALID_ARG;
  if (c->mask_token_id < 0 || c->mask_token_id >= c->vocab) return DFLASH_ERR_INVALID_ARG;
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta >= 0.f)) return DFLASH_ERR_INVALID_ARG;
  const int R = c->gamma + 1;
  if (c->ctx_capacity < R + 1) return DFLASH_ERR_INVALID_ARG;
  if (c->head_dim != 64 && c->head_dim != 128) return DFLASH_ERR_SHAPE;
  if (c->n_q_heads % c->n_kv_heads != 0) return DFLASH_ERR_SHAPE;
  if ((c->n_q_heads / c->n_kv_heads) * R > 128) return DFLASH_ERR_SHAPE;
  const int bk = c->dtype == DFLASH_BF16 ? 64 : 32;
  const long long kin = static_cast<long long>(c->n_taps) * c->d_target;
  if (c->d_model % kBM || c->d_model > 8192 || kin % bk || (c->n_q_heads * c->head_dim) % bk ||
      c->d_ffn % 64)
    return DFLASH_ERR_SHAPE;
  if (((c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim) % kBM) return DFLASH_ERR_SHAPE;
  if ((2 * c->n_kv_heads * c->head_dim) % kBM) return DFLASH_ERR_SHAPE;
  if (kin > (1LL << 30) || static_cast<long long>(c->vocab) * c->d_model > (1LL << 40))
    return DFLASH_ERR_SHAPE;
  return DFLASH_OK;
}

size_t dflash_param_bytes(const dflash_config* c, int kind) {
  if (dflash_check_config(c) != DFLASH_OK) return 0;
  const size_t es = elem_bytes(c);
  const size_t D = c->d_model, V = c->vocab, L = c->n_layers, F = c->d_ffn;
  const size_t HD = static_cast<size_t>(c->n_q_heads) * c->head_dim;
  const size_t nqkv = static_cast<size_t>(c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim;
  const size_t wc = D * c->n_taps * c->d_target * es;
  const size_t emb = V * D * es;
  const size_t head = V * D * es;
  const size_t layers = L * (nqkv * D + D * HD + 2 * F * D + D * F + 2 * D) * es;
  switch (kind) {
    case 0: return wc;
    case 1: return emb;
    case 2: return head;
    case 3: return layers;
    case 4: return wc + D * es + emb + head + D * es + layers;
  }
  return 0;
}

size_t dflash_kv_cache_bytes(const dflash_config* c) {
  if (dflash_check_config(c) != DFLASH_OK) return 0;
  return static_cast<size_t>(c->n_layers) * c->max_batch * c->n_kv_heads * c->ctx_capacity *
         c->head_dim * elem_bytes(c);
}

size_t dflash_workspace_bytes(const dflash_config* c, int max_rows) {
  if (dflash_check_config(c) != DFLASH_OK || max_rows < 0) return 0;
  const WsLayout L = ws_layout(c);
  return L.fixed + align256(static_cast<size_t>(max_rows) * row_ss_bytes_per_row(c));
}

dflash_status dflash_selftest_wait_timeout(int32_t* dev_status, dflash_stream_t stream) {
  if (dev_status == nullptr) return DFLASH_ERR_INVALID_ARG;
  dflash_status st = check_arch();
  if (st != DFLASH_OK) return st;
  return launch_wait_selftest(dev_status, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DFLASH_OK
             : DFLASH_ERR_CUDA;
}

dflash_status dflash_workspace_init(void* ws, size_t ws_bytes, dflash_stream_t stream) {
  if (ws == nullptr || ws_bytes == 0) return DFLASH_ERR_INVALID_ARG;
  if (cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  return DFLASH_OK;
}

dflash_status dflash_rope_tables(const dflash_config* c, int n_pos, float* host_cos, float* host_sin) {
  if (c == nullptr || host_cos == nullptr || host_sin == nullptr || n_pos < 0)
    return DFLASH_ERR_INVALID_ARG;
  if (c->head_dim < 2 || c->head_dim % 2) return DFLASH_ERR_SHAPE;
  const int half = c->head_dim / 2;
  for (int p = 0; p < n_pos; ++p) {
    for (int j = 0; j < half; ++j) {
      const double inv = c->rope_theta > 0.f ? pow(static_cast<double>(c->rope_theta), -2.0 * j / c->head_dim) : 0.0;
      const double ang = static_cast<double>(p) * inv;
      host_cos[static_cast<size_t>(p) * half + j] = static_cast<float>(cos(ang));
      host_sin[static_cast<size_t>(p) * half + j] = static_cast<float>(sin(ang));
    }
  }
  return DFLASH_OK;
}

}  // extern "C"

namespace {

void fill_from_plan(GemmArgs& g, const GemmPlan& p, int k) {
  g.k = k;
  g.group_m = p.group_m;
  g.bn = p.bn;
  g.n_sub = p.n_sub;
  g.kt_per_split = p.kt_per_split;
  g.splits = p.splits;
  g.m_tiles = p.m_tiles;
  g.n_tiles = p.n_tiles;
  if (g.a_tiles_per_z <= 0) g.a_tiles_per_z = p.m_tiles;
  if (g.b_tiles_per_z <= 0) g.b_tiles_per_z = p.n_tiles;
}

struct Ctx {
  const dflash_config* c;
  WsLayout L;
  void* ws;
  cudaStream_t s;
  int es;
  int sms;
  bool pdl;
  Tracer tr;
};

// One projection launch: A rows a_rows (weights when swap), B rows b_rows.
dflash_status run_gemm(Ctx& x, GemmArgs g, const CUtensorMap& amap, const CUtensorMap& bmap,
                       GemmPlan plan, double bytes, double flops) {
  fill_from_plan(g, plan, g.k);
  g.tf32 = x.c->dtype == DFLASH_F32;
  x.tr.before(DFLASH_K_GEMM, bytes, flops);
  const cudaError_t e = launch_gemm(amap, bmap, g, plan, x.s, x.pdl);
  x.tr.after();
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

Epi base_epi(const dflash_config* c) {
  Epi e{};
  e.out_bf16 = c->dtype == DFLASH_BF16 ? 1 : 0;
  e.max_batch = c->max_batch;
  e.n_q_heads = c->n_q_heads;
  e.n_kv_heads = c->n_kv_heads;
  e.head_dim = c->head_dim;
  e.ncap = c->ctx_capacity;
  e.reserve = c->gamma + 1;
  return e;
}

// A page view: both pools, a table, at least one page and the block's
// reserve within one sequence's pages.
bool pages_ok(const dflash_config* c, const dflash_kv_pages* p) {
  return p != nullptr && p->k_pool != nullptr && p->v_pool != nullptr && p->page_table != nullptr &&
         p->n_pages >= 1 && p->pages_per_seq >= 1 &&
         static_cast<long long>(p->pages_per_seq) * DFLASH_PAGE_KEYS >= c->gamma + 2;
}

bool trace_ok(const dflash_trace* t) {
  return t == nullptr || (t->events != nullptr && t->kinds != nullptr && t->bytes != nullptr &&
                          t->flops != nullptr && t->capacity >= 0);
}

// RoPE tables cover every position a sequence of capacity ncap can reach.
bool rope_ok(const dflash_config* c, const dflash_weights* w, int ncap) {
  if (c->rope_theta == 0.f) return true;
  return w->rope_cos != nullptr && w->rope_sin != nullptr && w->rope_positions >= ncap;
}

}  // namespace

extern "C" {

dflash_status dflash_linear(dflash_dtype dtype, const void* x, const void* w, float* y, int M, int N,
                            int K, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  if (dtype != DFLASH_BF16 && dtype != DFLASH_F32) return DFLASH_ERR_DTYPE;
  if (M < 0 || N < 0 || K <= 0) return DFLASH_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return DFLASH_OK;
  if (x == nullptr || w == nullptr || y == nullptr) return DFLASH_ERR_INVALID_ARG;
  const int es = dtype == DFLASH_BF16 ? 2 : 4;
  if (K % (128 / es)) return DFLASH_ERR_SHAPE;
  (void)ws;
  (void)ws_bytes;
  dflash_status st = check_arch();
  if (st != DFLASH_OK) return st;
  dflash_config cfg{};
  cfg.dtype = dtype;
  Ctx cx{&cfg, WsLayout{}, ws, reinterpret_cast<cudaStream_t>(stream), es, num_sms_of_current_device(),
         use_pdl(), Tracer{nullptr, nullptr}};
  GemmArgs g{};
  CUtensorMap amap, bmap;
  GemmPlan plan;
  const bool swap = M <= kMaxBN;
  if (swap) {
    plan = plan_gemm((N + kBM - 1) / kBM, M, K, es, cx.sms, true, true);
    if (!make_operand_map(&amap, w, es, K, N, 1, kBM) ||
        !make_operand_map(&bmap, x, es, K, M, 1, plan.bn / plan.n_sub))
      return DFLASH_ERR_ALIGN;
    g.swap = 1;
    g.a_weights = 1;
  } else {
    plan = plan_gemm((M + kBM - 1) / kBM, N, K, es, cx.sms, false, false);
    if (!make_operand_map(&amap, x, es, K, M, 1, kBM) ||
        !make_operand_map(&bmap, w, es, K, N, 1, plan.bn / plan.n_sub))
      return DFLASH_ERR_ALIGN;
  }
  g.k = K;
  g.m_rows = swap ? N : M;
  g.n_rows = swap ? M : N;
  g.epi.op = EPI_STORE;
  g.epi.out = y;
  g.epi.ld = N;
  g.epi.out_bf16 = 0;
  g.epi.n_tok = M;
  g.epi.n_feat = N;
  return run_gemm(cx, g, amap, bmap, plan, 0.0, 0.0);
}

dflash_status dflash_ctx_fuse(const dflash_config* c, const dflash_weights* w, const void* taps, int T,
                              void* h_ctx, void* ws, size_t ws_bytes, dflash_trace* trace,
                              dflash_stream_t stream) {
  dflash_status st = dflash_check_config(c);
  if (st != DFLASH_OK) return st;
  if (w == nullptr || T < 0) return DFLASH_ERR_INVALID_ARG;
  if (T == 0) return DFLASH_OK;
  if (taps == nullptr || h_ctx == nullptr || w->w_c == nullptr || w->g_c == nullptr ||
      !trace_ok(trace))
    return DFLASH_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c);
  if (ws == nullptr || ws_bytes < L.fixed + static_cast<size_t>(T) * row_ss_bytes_per_row(c))
    return DFLASH_ERR_WORKSPACE;
  if ((st = check_arch()) != DFLASH_OK) return st;
  const int es = elem_bytes(c), D = c->d_model, K = c->n_taps * c->d_target;
  Ctx cx{c, L, ws, reinterpret_cast<cudaStream_t>(stream), es, num_sms_of_current_device(), use_pdl(),
         Tracer{trace, reinterpret_cast<cudaStream_t>(stream)}};
  GemmArgs g{};
  CUtensorMap amap, bmap;
  GemmPlan plan;
  const bool swap = T <= kMaxBN;
  if (swap) {
    plan = plan_gemm(D / kBM, T, K, es, cx.sms, true, true);
    if (!make_operand_map(&amap, w->w_c, es, K, D, 1, kBM) ||
        !make_operand_map(&bmap, taps, es, K, T, 1, plan.bn / plan.n_sub))
      return DFLASH_ERR_ALIGN;
    g.swap = 1;
    g.a_weights = 1;
  } else {
    plan = plan_gemm((T + kBM - 1) / kBM, D, K, es, cx.sms, false, false);
    if (!make_operand_map(&amap, taps, es, K, T, 1, kBM) ||
        !make_operand_map(&bmap, w->w_c, es, K, D, 1, plan.bn / plan.n_sub))
      return DFLASH_ERR_ALIGN;
  }
  g.k = K;
  g.m_rows = swap ? D : T;
  g.n_rows = swap ? T : D;
  g.dev_status = nullptr;
  // u = W_c x stays fp32 in the workspace; the norm pass rounds once to cfg.dtype
  float* u32 = at<float>(ws, L.row_ss);
  float* row_ss = u32 + static_cast<size_t>(T) * D;
  g.epi = base_epi(c);
  g.epi.op = EPI_FUSE;
  g.epi.out = u32;
  g.epi.out_bf16 = 0;
  g.epi.ld = D;
  g.epi.n_tok = T;
  g.epi.n_feat = D;
  g.epi.row_ss = row_ss;
  g.epi.n_ss = D / kBM;
  const double bytes = (static_cast<double>(T) * K + static_cast<double>(D) * K + static_cast<double>(T) * D) * es;
  if ((st = run_gemm(cx, g, amap, bmap, plan, bytes, 2.0 * T * D * static_cast<double>(K))) != DFLASH_OK)
    return st;
  cx.tr.before(DFLASH_K_NORM, 2.0 * T * D * es, 0);
  const cudaError_t e = launch_fuse_norm(u32, h_ctx, row_ss, D / kBM, w->g_c, T, D, c->rms_eps,
                                         c->dtype == DFLASH_BF16, cx.s, cx.pdl);
  cx.tr.after();
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

static dflash_status kv_inject_impl(const dflash_config* c, const dflash_weights* w, const void* h_ctx,
                                    const int32_t* n_new, int B, int Tmax, int32_t* ctx_len, void* k_cache,
                                    void* v_cache, const dflash_kv_pages* pages, int32_t* dev_status, void* ws,
                                    size_t ws_bytes, dflash_trace* trace, dflash_stream_t stream) {
  dflash_status st = dflash_check_config(c);
  if (st != DFLASH_OK) return st;
  // capacity per sequence: the contiguous cache's, or the pages of its table
  const int ncap = pages != nullptr ? pages->pages_per_seq * DFLASH_PAGE_KEYS : c->ctx_capacity;
  if (w == nullptr || B < 0 || B > c->max_batch || Tmax < 0) return DFLASH_ERR_INVALID_ARG;
  if (B == 0 || Tmax == 0) return DFLASH_OK;
  if (h_ctx == nullptr || n_new == nullptr || ctx_len == nullptr || k_cache == nullptr ||
      v_cache == nullptr || dev_status == nullptr || w->w_qkv == nullptr || !rope_ok(c, w, ncap) ||
      !trace_ok(trace))
    return DFLASH_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c);
  if (ws == nullptr || ws_bytes < L.fixed) return DFLASH_ERR_WORKSPACE;
  if ((st = check_arch()) != DFLASH_OK) return st;
  const int es = elem_bytes(c), D = c->d_model;
  const int rows = B * Tmax;
  const int nqkv = (c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim;
  const int fpl = 2 * c->n_kv_heads * c->head_dim;
  Ctx cx{c, L, ws, reinterpret_cast<cudaStream_t>(stream), es, num_sms_of_current_device(), use_pdl(),
         Tracer{trace, reinterpret_cast<cudaStream_t>(stream)}};
  GemmArgs g{};
  CUtensorMap amap, bmap;
  GemmPlan plan;
  const bool swap = rows <= kMaxBN;
  if (swap) {
    plan = plan_gemm(c->n_layers * fpl / kBM, rows, D, es, cx.sms, true, true);
    if (!make_operand_map(&amap, w->w_qkv, es, D, nqkv, c->n_layers, kBM) ||
        !make_operand_map(&bmap, h_ctx, es, D, rows, 1, plan.bn / plan.n_sub))
      return DFLASH_ERR_ALIGN;
    g.swap = 1;
    g.a_weights = 1;
    g.a_row0 = c->n_q_heads * c->head_dim;
    g.a_tiles_per_z = fpl / kBM;
  } else {
    // feature tiles must not straddle layers
    const int cap = fpl % 512 == 0 ? 512 : (fpl % 256 == 0 ? 256 : kBM);
    plan = plan_gemm((rows + kBM - 1) / kBM, c->n_layers * fpl, D, es, cx.sms, false, false, cap);
    if (!make_operand_map(&amap, h_ctx, es, D, rows, 1, kBM) ||
        !make_operand_map(&bmap, w->w_qkv, es, D, nqkv, c->n_layers, plan.bn / plan.n_sub))
      return DFLASH_ERR_ALIGN;
    g.b_row0 = c->n_q_heads * c->head_dim;
    g.b_tiles_per_z = fpl / plan.bn;
  }
  g.k = D;
  g.m_rows = swap ? c->n_layers * fpl : rows;
  g.n_rows = swap ? rows : c->n_layers * fpl;
  g.dev_status = dev_status;
  g.epi = base_epi(c);
  g.epi.op = EPI_KV;
  g.epi.k_cache = k_cache;
  g.epi.v_cache = v_cache;
  g.epi.ncap = ncap;
  if (pages != nullptr) {
    g.epi.page_table = pages->page_table;
    g.epi.n_pages = pages->n_pages;
    g.epi.pages_per_seq = pages->pages_per_seq;
  }
  g.epi.ctx_len = ctx_len;
  g.epi.n_new = n_new;
  g.epi.rows_per_seq = Tmax;
  g.epi.feat_per_layer = fpl;
  g.epi.n_tok = rows;
  g.epi.n_feat = c->n_layers * fpl;
  g.epi.rope_cos = c->rope_theta > 0.f ? w->rope_cos : nullptr;
  g.epi.rope_sin = c->rope_theta > 0.f ? w->rope_sin : nullptr;
  g.epi.rope_positions = w->rope_positions;
  const double bytes = (static_cast<double>(rows) * D + static_cast<double>(c->n_layers) * fpl * D +
                        static_cast<double>(rows) * c->n_layers * fpl) * es;
  if ((st = run_gemm(cx, g, amap, bmap, plan, bytes, 2.0 * rows * c->n_layers * static_cast<double>(fpl) * D)) != DFLASH_OK)
    return st;
  cx.tr.before(DFLASH_K_NORM, 12.0 * B, 0);
  const cudaError_t e = launch_kv_advance(ctx_len, n_new, B, Tmax, ncap, c->gamma + 1, dev_status, cx.s,
                                          cx.pdl);
  cx.tr.after();
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

dflash_status dflash_kv_inject(const dflash_config* c, const dflash_weights* w, const void* h_ctx,
                               const int32_t* n_new, int B, int Tmax, int32_t* ctx_len, void* k_cache,
                               void* v_cache, int32_t* dev_status, void* ws, size_t ws_bytes,
                               dflash_trace* trace, dflash_stream_t stream) {
  return kv_inject_impl(c, w, h_ctx, n_new, B, Tmax, ctx_len, k_cache, v_cache, nullptr, dev_status, ws,
                        ws_bytes, trace, stream);
}

dflash_status dflash_kv_inject_paged(const dflash_config* c, const dflash_weights* w, const void* h_ctx,
                                     const int32_t* n_new, int B, int Tmax, int32_t* ctx_len,
                                     const dflash_kv_pages* pages, int32_t* dev_status, void* ws, size_t ws_bytes,
                                     dflash_trace* trace, dflash_stream_t stream) {
  if (!pages_ok(c, pages)) return DFLASH_ERR_INVALID_ARG;
  return kv_inject_impl(c, w, h_ctx, n_new, B, Tmax, ctx_len, pages->k_pool, pages->v_pool, pages, dev_status,
                        ws, ws_bytes, trace, stream);
}

}  // extern "C"

extern "C" {

static dflash_status draft_block_impl(const dflash_config* c, const dflash_weights* w, const int32_t* anchor,
                                      const int32_t* ids, const int32_t* ctx_len, const int32_t* gamma_b, int B,
                                      int max_ctx_hint, void* k_cache,
                                      void* v_cache, float temperature, uint64_t seed, int32_t* draft,
                                      float* logits_opt, float* layer_dump_opt, int32_t* dev_status, void* ws,
                                      size_t ws_bytes, dflash_trace* trace, dflash_stream_t stream,
                                      const dflash_kv_pages* pages = nullptr) {
  const int ncap = pages != nullptr ? pages->pages_per_seq * DFLASH_PAGE_KEYS : c->ctx_capacity;
  dflash_status st = dflash_check_config(c);
  if (st != DFLASH_OK) return st;
  if (w == nullptr || B < 1 || B > c->max_batch || max_ctx_hint < 0) return DFLASH_ERR_INVALID_ARG;
  if ((anchor == nullptr && ids == nullptr) || ctx_len == nullptr || k_cache == nullptr || v_cache == nullptr ||
      draft == nullptr || dev_status == nullptr || w->embed == nullptr || w->g_final == nullptr ||
      w->lm_head == nullptr || w->g_attn == nullptr || w->w_qkv == nullptr || w->w_o == nullptr ||
      w->g_ffn == nullptr || w->w_gateup == nullptr || w->w_down == nullptr || !rope_ok(c, w, ncap))
    return DFLASH_ERR_INVALID_ARG;
  if (!trace_ok(trace)) return DFLASH_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c);
  if (ws == nullptr || ws_bytes < L.fixed) return DFLASH_ERR_WORKSPACE;
  if ((st = check_arch()) != DFLASH_OK) return st;

  const int es = elem_bytes(c);
  const int bf16 = c->dtype == DFLASH_BF16;
  const int D = c->d_model, F = c->d_ffn, V = c->vocab, Lyr = c->n_layers;
  const int R = c->gamma + 1, rows = B * R, nmask = B * c->gamma;
  const int HD = c->n_q_heads * c->head_dim;
  const int nqkv = (c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim;
  Ctx cx{c, L, ws, reinterpret_cast<cudaStream_t>(stream), es, num_sms_of_current_device(), use_pdl(),
         Tracer{trace, reinterpret_cast<cudaStream_t>(stream)}};
  float* h = at<float>(ws, L.h);
  void* xn = at<void>(ws, L.xn);
  void* q = at<void>(ws, L.q);
  void* ao = at<void>(ws, L.attn_o);
  void* act = at<void>(ws, L.act);
  void* z = at<void>(ws, L.z);
  unsigned long long* keys = at<unsigned long long>(ws, L.lm_keys);
  const double row_bytes = static_cast<double>(rows) * D * 4;

  // Skinny projection plans (tokens ride along as the MMA's N). bf16 models
  // feed each projection hi and lo halves of its activation (split = true).
  const bool split = bf16 != 0;
  const int rows_max = c->max_batch * R, nmask_max = c->max_batch * c->gamma;
  const int parts = split ? 2 : 1;
  GemmPlan p_qkv = plan_gemm(nqkv / kBM, rows, D, es, cx.sms, true, true, kMaxBN, split, true);
  const GemmPlan p_o = plan_gemm(D / kBM, rows, HD, es, cx.sms, true, true, kMaxBN, split, true);
  GemmPlan p_gu = plan_gemm(F / 64, rows, D, es, cx.sms, true, true, kMaxBN, split, true);
  if (p_qkv.b_split != p_gu.b_split) {  // both read the same normed activations
    p_qkv = plan_gemm(nqkv / kBM, rows, D, es, cx.sms, true, true, kMaxBN, false, true);
    p_gu = plan_gemm(F / 64, rows, D, es, cx.sms, true, true, kMaxBN, false, true);
  }
  const GemmPlan p_dn = plan_gemm(D / kBM, rows, F, es, cx.sms, true, true, kMaxBN, split, true);
  const GemmPlan p_lm = plan_gemm((V + kBM - 1) / kBM, nmask, D, es, cx.sms, false, true, kMaxBN, split, true);

  // B boxes bring the valid token rows alone (hi and lo rows when the plan
  // packs split operands) when one box spans the tile
  auto box_of = [](const GemmPlan& p, int n) {
    return p.b_split ? 2 * n : (p.n_sub == 1 && p.n_tiles == 1 ? n : p.bn / p.n_sub);
  };
  CUtensorMap m_qkv, m_o, m_gu, m_dn, m_lm, m_xn, m_ao, m_act, m_z;
  bool ok = make_operand_map(&m_qkv, w->w_qkv, es, D, nqkv, Lyr, kBM) &&
            make_operand_map(&m_o, w->w_o, es, HD, D, Lyr, kBM) &&
            make_operand_map(&m_gu, w->w_gateup, es, D, 2 * F, Lyr, 64) &&
            make_operand_map(&m_dn, w->w_down, es, F, D, Lyr, kBM) &&
            make_operand_map(&m_lm, w->lm_head, es, D, V, 1, kBM) &&
            make_operand_map(&m_xn, xn, es, D, parts * rows_max, 1, box_of(p_qkv, rows)) &&
            make_operand_map(&m_ao, ao, es, HD, parts * rows_max, 1, box_of(p_o, rows)) &&
            make_operand_map(&m_act, act, es, F, parts * rows_max, 1, box_of(p_dn, rows)) &&
            make_operand_map(&m_z, z, es, D, parts * nmask_max, 1, box_of(p_lm, nmask));
  if (!ok) return DFLASH_ERR_ALIGN;
  CUtensorMap m_xn_gu;  // same buffer, box of the gate|up plan
  if (!make_operand_map(&m_xn_gu, xn, es, D, parts * rows_max, 1, box_of(p_gu, rows)))
    return DFLASH_ERR_ALIGN;
  // Each activation buffer carries lo = x - bf16(x) rows right after its hi
  // rows when its consuming projection takes split operands (the planner
  // decides per shape), so that one box brings both.
  const bool s_xn = p_qkv.b_split && p_gu.b_split, s_ao = p_o.b_split, s_act = p_dn.b_split,
             s_z = p_lm.b_split;
  const size_t xn_lo = s_xn ? static_cast<size_t>(rows) * D : 0;
  const size_t ao_lo = s_ao ? static_cast<size_t>(rows) * HD : 0;
  const size_t act_lo = s_act ? static_cast<size_t>(rows) * F : 0;
  const size_t z_lo = s_z ? static_cast<size_t>(nmask) * D : 0;
  auto pack_of = [&](bool on, int n) { return on ? n : 0; };

  auto fail = [](cudaError_t e) { return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA; };

  float* ss = at<float>(ws, L.ss);
  const int n_ss = D / kBM;
  // RMSNorm is folded into the projections: the producer of h writes g (.) h and
  // per-token sums of squares; the consuming GEMM scales by rstd per token.
  auto fold_in = [&](Epi& e) {
    e.ss_in = ss;
    e.n_ss = n_ss;
    e.d_model = D;
    e.eps = c->rms_eps;
  };
  auto fold_out = [&](Epi& e, void* xg, const void* gain, int mask_rows) {
    e.xg_out = xg;
    e.lo_off = mask_rows ? z_lo : xn_lo;
    e.xg_gain = gain;
    e.xg_bf16 = bf16;
    e.ss_out = ss;
    e.n_ss = n_ss;
    e.d_model = D;
    e.xg_mask_rows = mask_rows;
    e.gamma = c->gamma;
    e.rows_per_seq = R;
  };
  auto gain_of = [&](const void* g, int l) {
    return static_cast<const void*>(static_cast<const uint8_t*>(g) + static_cast<size_t>(l) * D * es);
  };

  cx.tr.before(DFLASH_K_NORM, row_bytes + static_cast<double>(rows) * D * es, 0);
  st = fail(launch_embed(w->embed, anchor, ids, c->mask_token_id, B, R, D, V, bf16, h, gain_of(w->g_attn, 0),
                         xn, xn_lo, ss, dev_status, cx.s, cx.pdl));
  cx.tr.after();
  if (st != DFLASH_OK) return st;
  if (layer_dump_opt != nullptr &&
      launch_copy_f32(layer_dump_opt, h, static_cast<size_t>(rows) * D, cx.s, cx.pdl) != cudaSuccess)
    return DFLASH_ERR_CUDA;

  int a_splits = 1, a_chunk = 0, a_global = 0;
  plan_attention(B, R, c->n_q_heads, c->n_kv_heads, c->head_dim, max_ctx_hint, ncap, cx.sms,
                 &a_splits, &a_chunk, &a_global);

  for (int l = 0; l < Lyr; ++l) {
    // Q/K/V projection of RMSNorm(h): RoPE; block K/V into the cache scratch rows
    {
      GemmArgs g{};
      g.k = D; g.m_rows = nqkv; g.n_rows = rows; g.swap = 1; g.a_weights = 1; g.a_z0 = l;
      g.b_pack = pack_of(s_xn, rows); g.b_box_rows = box_of(p_qkv, rows);
      g.dev_status = dev_status;
      g.epi = base_epi(c);
      g.epi.op = EPI_QKV; g.epi.out = q; g.epi.ld = HD; g.epi.n_tok = rows; g.epi.n_feat = nqkv;
      g.epi.k_cache = k_cache; g.epi.v_cache = v_cache; g.epi.ctx_len = ctx_len;
      g.epi.ncap = ncap;
      if (pages != nullptr) {
        g.epi.page_table = pages->page_table;
        g.epi.n_pages = pages->n_pages;
        g.epi.pages_per_seq = pages->pages_per_seq;
      }
      g.epi.rows_per_seq = R; g.epi.layer = l;
      g.epi.rope_cos = c->rope_theta > 0.f ? w->rope_cos : nullptr;
      g.epi.rope_sin = c->rope_theta > 0.f ? w->rope_sin : nullptr;
      g.epi.rope_positions = w->rope_positions;
      fold_in(g.epi);
      const double b = (static_cast<double>(nqkv) * D + static_cast<double>(rows) * (D + nqkv)) * es;
      if ((st = run_gemm(cx, g, m_qkv, m_xn, p_qkv, b, 2.0 * rows * nqkv * static_cast<double>(D))) != DFLASH_OK)
        return st;
    }
    // attention over [injected context ; block]
    {
      AttnArgs a{};
      a.q = q;
      a.k_cache = k_cache;
      a.v_cache = v_cache;
      a.layer = l;
      a.n_layers = Lyr;
      a.ctx_len = ctx_len; a.gamma_b = gamma_b; a.out = ao;
      a.out_lo_off = ao_lo;
      a.dev_status = dev_status;
      a.B = B; a.R = R; a.n_q_heads = c->n_q_heads; a.n_kv_heads = c->n_kv_heads;
      a.head_dim = c->head_dim; a.ncap = ncap; a.max_batch = c->max_batch;
      if (pages != nullptr) {
        a.page_table = pages->page_table;
        a.n_pages = pages->n_pages;
        a.pages_per_seq = pages->pages_per_seq;
      }
      a.splits = a_splits; a.chunk = a_chunk; a.bf16 = bf16;
      a.merge_global = a_global;
      a.partials = at<float>(cx.ws, cx.L.attn_part);
      const double kvb = 2.0 * B * c->n_kv_heads * static_cast<double>(max_ctx_hint + R) * c->head_dim * es;
      const double fl = 4.0 * B * c->n_q_heads * R * static_cast<double>(max_ctx_hint + R) * c->head_dim;
      cx.tr.before(DFLASH_K_ATTN, kvb + 2.0 * rows * HD * es, fl);
      st = fail(launch_attention(a, cx.s, cx.pdl));
      cx.tr.after();
      if (st != DFLASH_OK) return st;
      if (bf16 && a.splits > 1 && a.merge_global) {   // its merge: time, no algorithmic bytes
        cx.tr.before(DFLASH_K_ATTN, 0.0, 0.0);
        st = fail(launch_attention_merge(a, cx.s, cx.pdl));
        cx.tr.after();
        if (st != DFLASH_OK) return st;
      }
    }
    // output projection + residual; emits g_ffn (.) h and sums of squares
    {
      GemmArgs g{};
      g.k = HD; g.m_rows = D; g.n_rows = rows; g.swap = 1; g.a_weights = 1; g.a_z0 = l;
      g.b_pack = pack_of(s_ao, rows); g.b_box_rows = box_of(p_o, rows);
      g.dev_status = dev_status;
      g.epi = base_epi(c);
      g.epi.op = EPI_ADD_F32; g.epi.out = h; g.epi.ld = D; g.epi.n_tok = rows; g.epi.n_feat = D;
      fold_out(g.epi, xn, gain_of(w->g_ffn, l), 0);
      const double b = static_cast<double>(D) * HD * es + static_cast<double>(rows) * HD * es + 2.0 * row_bytes;
      if ((st = run_gemm(cx, g, m_o, m_ao, p_o, b, 2.0 * rows * D * static_cast<double>(HD))) != DFLASH_OK)
        return st;
    }
    // gate|up of RMSNorm(h) + SwiGLU
    {
      GemmArgs g{};
      g.k = D; g.m_rows = 2 * F; g.n_rows = rows; g.swap = 1; g.a_weights = 1; g.a_z0 = l;
      g.a_gateup = F;
      g.b_pack = pack_of(s_xn, rows); g.b_box_rows = box_of(p_gu, rows);
      g.dev_status = dev_status;
      g.epi = base_epi(c);
      g.epi.op = EPI_SWIGLU; g.epi.out = act; g.epi.ld = F; g.epi.n_tok = rows; g.epi.n_feat = F;
      g.epi.lo_off = act_lo;
      fold_in(g.epi);
      const double b = (2.0 * F * D + static_cast<double>(rows) * (D + F)) * es;
      if ((st = run_gemm(cx, g, m_gu, m_xn_gu, p_gu, b, 4.0 * rows * F * static_cast<double>(D))) != DFLASH_OK)
        return st;
    }
    // down + residual; emits the next layer's g_attn (.) h, or for the last
    // layer the final norm's g_final (.) h of the mask rows
    {
      GemmArgs g{};
      g.k = F; g.m_rows = D; g.n_rows = rows; g.swap = 1; g.a_weights = 1; g.a_z0 = l;
      g.b_pack = pack_of(s_act, rows); g.b_box_rows = box_of(p_dn, rows);
      g.dev_status = dev_status;
      g.epi = base_epi(c);
      g.epi.op = EPI_ADD_F32; g.epi.out = h; g.epi.ld = D; g.epi.n_tok = rows; g.epi.n_feat = D;
      if (l + 1 < Lyr)
        fold_out(g.epi, xn, gain_of(w->g_attn, l + 1), 0);
      else
        fold_out(g.epi, z, w->g_final, 1);
      const double b = static_cast<double>(D) * F * es + static_cast<double>(rows) * F * es + 2.0 * row_bytes;
      if ((st = run_gemm(cx, g, m_dn, m_act, p_dn, b, 2.0 * rows * D * static_cast<double>(F))) != DFLASH_OK)
        return st;
    }
    if (layer_dump_opt != nullptr &&
        launch_copy_f32(layer_dump_opt + static_cast<size_t>(l + 1) * rows * D, h,
                        static_cast<size_t>(rows) * D, cx.s, cx.pdl) != cudaSuccess)
      return DFLASH_ERR_CUDA;
  }
  // LM head of RMSNorm(h[mask rows]) with fused argmax
  {
    GemmArgs g{};
    g.k = D; g.m_rows = V; g.n_rows = nmask; g.swap = 1; g.a_weights = 1;
    g.b_pack = pack_of(s_z, nmask); g.b_box_rows = box_of(p_lm, nmask);
    g.dev_status = dev_status;
    g.epi = base_epi(c);
    g.epi.op = EPI_ARGMAX; g.epi.out = logits_opt; g.epi.ld = V; g.epi.n_tok = nmask; g.epi.n_feat = V;
    g.epi.keys = keys;
    g.epi.keys_ld = (V + kBM - 1) / kBM;
    g.epi.gamma = c->gamma;
    g.epi.temperature = temperature;
    g.epi.seed = seed;
    fold_in(g.epi);
    const double b = (static_cast<double>(V) * D + static_cast<double>(nmask) * D) * es;
    if ((st = run_gemm(cx, g, m_lm, m_z, p_lm, b, 2.0 * nmask * V * static_cast<double>(D))) != DFLASH_OK)
      return st;
  }
  cx.tr.before(DFLASH_K_ARGMAX, nmask * 12.0, 0);
  st = fail(launch_argmax_finalize(keys, (V + kBM - 1) / kBM, (V + kBM - 1) / kBM, nmask, c->gamma, gamma_b, draft,
                                   cx.s, cx.pdl));
  cx.tr.after();
  return st;
}

dflash_status dflash_draft_block(const dflash_config* c, const dflash_weights* w, const int32_t* anchor,
                                 const int32_t* ctx_len, int B, int max_ctx_hint, void* k_cache,
                                 void* v_cache, int32_t* draft, float* logits_opt,
                                 float* layer_dump_opt, int32_t* dev_status, void* ws, size_t ws_bytes,
                                 dflash_trace* trace, dflash_stream_t stream) {
  return draft_block_impl(c, w, anchor, nullptr, ctx_len, nullptr, B, max_ctx_hint, k_cache, v_cache, 0.f, 0, draft,
                          logits_opt, layer_dump_opt, dev_status, ws, ws_bytes, trace, stream);
}

dflash_status dflash_draft_block_paged(const dflash_config* c, const dflash_weights* w, const int32_t* anchor,
                                       const int32_t* ctx_len, int B, int max_ctx_hint, const dflash_kv_pages* pages,
                                       int32_t* draft, float* logits_opt, int32_t* dev_status, void* ws,
                                       size_t ws_bytes, dflash_trace* trace, dflash_stream_t stream) {
  if (!pages_ok(c, pages)) return DFLASH_ERR_INVALID_ARG;
  return draft_block_impl(c, w, anchor, nullptr, ctx_len, nullptr, B, max_ctx_hint, pages->k_pool, pages->v_pool,
                          0.f, 0, draft, logits_opt, nullptr, dev_status, ws, ws_bytes, trace, stream, pages);
}

dflash_status dflash_draft_block_dyn(const dflash_config* c, const dflash_weights* w, const int32_t* anchor,
                                     const int32_t* ctx_len, const int32_t* gamma_b, int B, int max_ctx_hint,
                                     void* k_cache, void* v_cache, int32_t* draft, float* logits_opt,
                                     int32_t* dev_status, void* ws, size_t ws_bytes, dflash_trace* trace,
                                     dflash_stream_t stream) {
  if (gamma_b == nullptr) return DFLASH_ERR_INVALID_ARG;
  return draft_block_impl(c, w, anchor, nullptr, ctx_len, gamma_b, B, max_ctx_hint, k_cache, v_cache, 0.f, 0, draft,
                          logits_opt, nullptr, dev_status, ws, ws_bytes, trace, stream);
}

dflash_status dflash_draft_block_ids(const dflash_config* c, const dflash_weights* w, const int32_t* ids,
                                     const int32_t* ctx_len, int B, int max_ctx_hint, void* k_cache,
                                     void* v_cache, int32_t* draft, float* logits_opt, int32_t* dev_status,
                                     void* ws, size_t ws_bytes, dflash_trace* trace, dflash_stream_t stream) {
  if (ids == nullptr) return DFLASH_ERR_INVALID_ARG;
  return draft_block_impl(c, w, nullptr, ids, ctx_len, nullptr, B, max_ctx_hint, k_cache, v_cache, 0.f, 0, draft,
                          logits_opt, nullptr, dev_status, ws, ws_bytes, trace, stream);
}

dflash_status dflash_unmask_step(const dflash_config* c, const float* logits, const int32_t* draft, int32_t* ids,
                                 int B, int steps_left, void* ws, size_t ws_bytes, dflash_trace* trace,
                                 dflash_stream_t stream) {
  dflash_status st = dflash_check_config(c);
  if (st != DFLASH_OK) return st;
  if (logits == nullptr || draft == nullptr || ids == nullptr || B < 1 || B > c->max_batch || steps_left < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (!trace_ok(trace)) return DFLASH_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c);
  if (ws == nullptr || ws_bytes < L.fixed) return DFLASH_ERR_WORKSPACE;
  if ((st = check_arch()) != DFLASH_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Tracer tr{trace, s};
  tr.before(DFLASH_K_VERIFY, static_cast<double>(B) * c->gamma * c->vocab * 4, 0);
  const cudaError_t e = launch_unmask_step(logits, draft, B, c->gamma, c->vocab, c->mask_token_id, steps_left,
                                           at<void>(ws, L.samp), ids, s, use_pdl());
  tr.after();
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

dflash_status dflash_draft_block_iter(const dflash_config* c, const dflash_weights* w, const int32_t* anchor,
                                      const int32_t* ctx_len, int B, int max_ctx_hint, void* k_cache,
                                      void* v_cache, int n_steps, int32_t* ids, int32_t* draft, float* logits,
                                      int32_t* dev_status, void* ws, size_t ws_bytes, dflash_trace* trace,
                                      dflash_stream_t stream) {
  dflash_status st = dflash_check_config(c);
  if (st != DFLASH_OK) return st;
  if (anchor == nullptr || ids == nullptr || draft == nullptr || logits == nullptr || B < 1 ||
      B > c->max_batch || n_steps < 1 || n_steps > c->gamma)
    return DFLASH_ERR_INVALID_ARG;
  if ((st = check_arch()) != DFLASH_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (launch_ids_init(anchor, c->mask_token_id, B, c->gamma + 1, ids, s, use_pdl()) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  for (int step = 0; step < n_steps; ++step) {
    st = draft_block_impl(c, w, nullptr, ids, ctx_len, nullptr, B, max_ctx_hint, k_cache, v_cache, 0.f, 0, draft,
                          logits, nullptr, dev_status, ws, ws_bytes, trace, stream);
    if (st != DFLASH_OK) return st;
    st = dflash_unmask_step(c, logits, draft, ids, B, n_steps - step, ws, ws_bytes, trace, stream);
    if (st != DFLASH_OK) return st;
  }
  return launch_ids_to_draft(ids, B, c->gamma, draft, s, use_pdl()) == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

dflash_status dflash_draft_block_sample(const dflash_config* c, const dflash_weights* w,
                                        const int32_t* anchor, const int32_t* ctx_len, int B,
                                        int max_ctx_hint, void* k_cache, void* v_cache, float temperature,
                                        uint64_t seed, int32_t* draft, float* logits,
                                        int32_t* dev_status, void* ws, size_t ws_bytes,
                                        dflash_trace* trace, dflash_stream_t stream) {
  if (!(temperature > 0.f) || !std::isfinite(temperature) || logits == nullptr) return DFLASH_ERR_INVALID_ARG;
  return draft_block_impl(c, w, anchor, nullptr, ctx_len, nullptr, B, max_ctx_hint, k_cache, v_cache, temperature, seed,
                          draft, logits, nullptr, dev_status, ws, ws_bytes, trace, stream);
}

dflash_status dflash_verify_sample(const dflash_config* c, const void* target_logits,
                                   dflash_dtype logits_dtype, const float* draft_logits,
                                   const int32_t* draft, int B, float temperature, uint64_t seed,
                                   int32_t* tau, int32_t* committed, int32_t* next_anchor, void* ws,
                                   size_t ws_bytes, dflash_trace* trace, dflash_stream_t stream) {
  dflash_status st = dflash_check_config(c);
  if (st != DFLASH_OK) return st;
  if (logits_dtype != DFLASH_BF16 && logits_dtype != DFLASH_F32) return DFLASH_ERR_DTYPE;
  if (B < 1 || B > c->max_batch || target_logits == nullptr || draft_logits == nullptr ||
      draft == nullptr || tau == nullptr || committed == nullptr || next_anchor == nullptr ||
      !(temperature > 0.f) || !std::isfinite(temperature))
    return DFLASH_ERR_INVALID_ARG;
  if (!trace_ok(trace)) return DFLASH_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c);
  if (ws == nullptr || ws_bytes < L.fixed) return DFLASH_ERR_WORKSPACE;
  if ((st = check_arch()) != DFLASH_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Tracer tr{trace, s};
  const int R = c->gamma + 1;
  // target rows once and drafter rows once for the statistics, then row a of each for the draw
  const double row = static_cast<double>(c->vocab);
  const double bytes = B * (R * row * (logits_dtype == DFLASH_BF16 ? 2 : 4) + c->gamma * row * 4 +
                            row * ((logits_dtype == DFLASH_BF16 ? 2 : 4) + 4));
  tr.before(DFLASH_K_VERIFY, bytes, 0);
  const cudaError_t e = launch_sample_verify(target_logits, logits_dtype == DFLASH_BF16, draft_logits, draft,
                                             B, c->gamma, c->vocab, temperature, seed, at<void>(ws, L.samp),
                                             tau, committed, next_anchor, s, use_pdl());
  tr.after();
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

dflash_status dflash_attention(const dflash_config* c, const void* q, const int32_t* ctx_len, int B,
                               int max_ctx_hint, int layer, const void* k_cache, const void* v_cache,
                               void* out, int32_t* dev_status, void* ws, size_t ws_bytes,
                               dflash_trace* trace, dflash_stream_t stream) {
  dflash_status st = dflash_check_config(c);
  if (st != DFLASH_OK) return st;
  if (B < 1 || B > c->max_batch || max_ctx_hint < 0 || layer < 0 || layer >= c->n_layers || q == nullptr ||
      ctx_len == nullptr || k_cache == nullptr || v_cache == nullptr || out == nullptr || dev_status == nullptr ||
      !trace_ok(trace))
    return DFLASH_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c);
  if (ws == nullptr || ws_bytes < L.fixed) return DFLASH_ERR_WORKSPACE;
  if ((st = check_arch()) != DFLASH_OK) return st;
  const int R = c->gamma + 1, es = elem_bytes(c);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  AttnArgs a{};
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.layer = layer;
  a.n_layers = c->n_layers;
  a.ctx_len = ctx_len;
  a.out = out;
  a.dev_status = dev_status;
  a.B = B; a.R = R; a.n_q_heads = c->n_q_heads; a.n_kv_heads = c->n_kv_heads;
  a.head_dim = c->head_dim; a.ncap = c->ctx_capacity; a.max_batch = c->max_batch;
  a.bf16 = c->dtype == DFLASH_BF16;
  plan_attention(B, R, c->n_q_heads, c->n_kv_heads, c->head_dim, max_ctx_hint, c->ctx_capacity,
                 num_sms_of_current_device(), &a.splits, &a.chunk, &a.merge_global);
  a.partials = at<float>(ws, L.attn_part);
  Tracer tr{trace, s};
  const double kvb = 2.0 * B * c->n_kv_heads * static_cast<double>(max_ctx_hint + R) * c->head_dim * es;
  const double fl = 4.0 * B * c->n_q_heads * R * static_cast<double>(max_ctx_hint + R) * c->head_dim;
  tr.before(DFLASH_K_ATTN, kvb + 2.0 * B * R * c->n_q_heads * c->head_dim * es, fl);
  cudaError_t e = launch_attention(a, s, use_pdl());
  tr.after();
  if (e == cudaSuccess && a.bf16 && a.splits > 1 && a.merge_global) {
    tr.before(DFLASH_K_ATTN, 0.0, 0.0);
    e = launch_attention_merge(a, s, use_pdl());
    tr.after();
  }
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

static dflash_status verify_accept_impl(const dflash_config* c, const void* target_logits,
                                        dflash_dtype logits_dtype, const int32_t* draft,
                                        const int32_t* gamma_b, int B, int32_t* tau,
                                   int32_t* committed, int32_t* next_anchor, void* ws, size_t ws_bytes,
                                   dflash_trace* trace, dflash_stream_t stream) {
  dflash_status st = dflash_check_config(c);
  if (st != DFLASH_OK) return st;
  if (logits_dtype != DFLASH_BF16 && logits_dtype != DFLASH_F32) return DFLASH_ERR_DTYPE;
  if (B < 1 || B > c->max_batch || target_logits == nullptr || draft == nullptr || tau == nullptr ||
      committed == nullptr || next_anchor == nullptr)
    return DFLASH_ERR_INVALID_ARG;
  if (!trace_ok(trace)) return DFLASH_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(c);
  if (ws == nullptr || ws_bytes < L.fixed) return DFLASH_ERR_WORKSPACE;
  if ((st = check_arch()) != DFLASH_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Tracer tr{trace, s};
  const int R = c->gamma + 1;
  const double bytes = static_cast<double>(B) * R * c->vocab * (logits_dtype == DFLASH_BF16 ? 2 : 4);
  tr.before(DFLASH_K_VERIFY, bytes, 0);
  const cudaError_t e = launch_verify(target_logits, logits_dtype == DFLASH_BF16, draft, gamma_b, B, c->gamma,
                                      c->vocab, tau, committed, next_anchor,
                                      at<unsigned long long>(ws, L.v_keys), at<int>(ws, L.v_count), s,
                                      use_pdl());
  tr.after();
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

dflash_status dflash_verify_accept(const dflash_config* c, const void* target_logits,
                                   dflash_dtype logits_dtype, const int32_t* draft, int B, int32_t* tau,
                                   int32_t* committed, int32_t* next_anchor, void* ws, size_t ws_bytes,
                                   dflash_trace* trace, dflash_stream_t stream) {
  return verify_accept_impl(c, target_logits, logits_dtype, draft, nullptr, B, tau, committed, next_anchor, ws,
                            ws_bytes, trace, stream);
}

dflash_status dflash_verify_accept_dyn(const dflash_config* c, const void* target_logits,
                                       dflash_dtype logits_dtype, const int32_t* draft, const int32_t* gamma_b,
                                       int B, int32_t* tau, int32_t* committed, int32_t* next_anchor,
                                       void* ws, size_t ws_bytes, dflash_trace* trace,
                                       dflash_stream_t stream) {
  if (gamma_b == nullptr) return DFLASH_ERR_INVALID_ARG;
  return verify_accept_impl(c, target_logits, logits_dtype, draft, gamma_b, B, tau, committed, next_anchor, ws,
                            ws_bytes, trace, stream);
}

}  // extern "C"
