// Context attention: dispatch, split planning, and the fp32 path.
//
// Every block row of every query head attends to all ctx_len[b] + R keys of
// its KV head, with no mask (bidirectional inside the block; "KV Injection
// 메커니즘" K_i/V_i equations of "DFlash: Block Diffusion for Flash Speculative
// Decoding 논문 정리", and §3.2 of the marsggbo DFlash page). bf16 drafters run
// on the tcgen05 kernel of attention_tc.cu; fp32 drafters (small test-size
// models) run the CUDA-core kernel below.
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"

namespace dfl {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
// split-KV CTAs of one (sequence, KV head) form one cluster; at one CTA per
// SM, clusters above 12 CTAs measured slower (fewer fit in a GPC at once)
constexpr int kMaxAttnCluster = 12;

// fp32 path (small fp32 drafters): one CTA per (block row, query head, sequence),
// each thread an online-softmax state over a strided subset of keys, merged in a
// fixed order through shared memory.
template <int DH>
__global__ void __launch_bounds__(128) attn_f32_kernel(const AttnArgs p) {
  __shared__ float s_o[128][DH + 1];
  __shared__ float s_m[128], s_l[128];
  const int i = blockIdx.x, hq = blockIdx.y, b = blockIdx.z;
  const int G = p.n_q_heads / p.n_kv_heads, kvh = hq / G;
  pdl_launch_dependents();
  pdl_wait();
  const int r_b = p.gamma_b == nullptr ? p.R : min(max(p.gamma_b[b], 1), p.R - 1) + 1;
  const int n_keys = p.ctx_len[b] + r_b;
  const size_t hq_stride = static_cast<size_t>(p.n_q_heads) * DH;
  const float* q = reinterpret_cast<const float*>(p.q) + (static_cast<size_t>(b) * p.R + i) * hq_stride + hq * DH;
  const float* kg = reinterpret_cast<const float*>(p.k_cache);   // this layer's cache or page pool
  const float* vg = reinterpret_cast<const float*>(p.v_cache);
  // element offset of key j (paged: through the page table)
  auto key_off = [&](int j) -> size_t {
    if (p.page_table == nullptr)
      return ((static_cast<size_t>(b) * p.n_kv_heads + kvh) * p.ncap + j) * DH;
    int pg = p.page_table[static_cast<size_t>(b) * p.pages_per_seq + j / kPageKeys];
    if (pg < 0 || pg >= p.n_pages) pg = 0;  // reported by whoever wrote the row
    return ((static_cast<size_t>(pg) * p.n_kv_heads + kvh) * kPageKeys + (j % kPageKeys)) * DH;
  };
  float qv[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) qv[d] = q[d];
  const float scale = rsqrtf(static_cast<float>(DH)) * kLog2e;
  float m = -INFINITY, l = 0.f, o[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) o[d] = 0.f;
  for (int j = threadIdx.x; j < n_keys; j += blockDim.x) {
    const size_t off = key_off(j);
    const float* kr = kg + off;
    float sdot = 0.f;
#pragma unroll
    for (int d = 0; d < DH; ++d) sdot += qv[d] * kr[d];
    sdot *= scale;
    const float mn = fmaxf(m, sdot);
    const float al = m == -INFINITY ? 0.f : exp2f(m - mn);
    const float pj = exp2f(sdot - mn);
    l = l * al + pj;
    const float* vr = vg + off;
#pragma unroll
    for (int d = 0; d < DH; ++d) o[d] = o[d] * al + pj * vr[d];
    m = mn;
  }
  s_m[threadIdx.x] = m;
  s_l[threadIdx.x] = l;
#pragma unroll
  for (int d = 0; d < DH; ++d) s_o[threadIdx.x][d] = o[d];
  __syncthreads();
  if (threadIdx.x < DH) {
    const int d = threadIdx.x;
    float M = -INFINITY;
    for (int t = 0; t < blockDim.x; ++t)
      if (s_l[t] > 0.f) M = fmaxf(M, s_m[t]);
    float L = 0.f, acc = 0.f;
    for (int t = 0; t < blockDim.x; ++t) {
      if (!(s_l[t] > 0.f)) continue;
      const float w = exp2f(s_m[t] - M);
      L += s_l[t] * w;
      acc += s_o[t][d] * w;
    }
    reinterpret_cast<float*>(p.out)[(static_cast<size_t>(b) * p.R + i) * hq_stride + hq * DH + d] =
        L > 0.f ? acc / L : 0.f;
  }
}

}  // namespace

void plan_attention(int B, int R, int Hq, int Hkv, int Dh, int max_ctx, int ncap, int num_sms,
                    int* splits, int* chunk, int* merge_global) {
  const int n_keys = (max_ctx < ncap ? max_ctx : ncap) + R;
  const int per_seq = B * Hkv > 0 ? B * Hkv : 1;
  const int tiles = (n_keys + 127) / 128;
  // Long contexts with few (sequence, KV head) pairs: a cluster of at most
  // kMaxAttnCluster splits per pair would leave SMs idle, so take one split
  // per SM (each at least two 128-key tiles) and merge through the workspace.
  const int sms = num_sms > 0 ? num_sms : 1;
  int wide = sms / per_seq;
  if (wide > kAttnMaxSlots / per_seq) wide = kAttnMaxSlots / per_seq;
  if (wide > tiles / 2) wide = tiles / 2;
  int sp, c;
  bool global = wide > kMaxAttnCluster;
  if (const char* e = getenv("DFLASH_ATTN_SPLITS")) {   // tuning override
    sp = atoi(e);
    if (sp < 1) sp = 1;
    if (sp > kAttnMaxSlots / per_seq) sp = kAttnMaxSlots / per_seq < 1 ? 1 : kAttnMaxSlots / per_seq;
    global = sp > kMaxAttnCluster;
  } else if (global) {
    sp = wide;
  } else {
    int per_sm = 2;   // ~2 CTAs per SM in total
    if (const char* e = getenv("DFLASH_ATTN_CTAS_PER_SM")) per_sm = atoi(e) > 0 ? atoi(e) : 1;   // tuning override
    sp = (per_sm * sms + per_seq - 1) / per_seq;
    if (sp > kMaxAttnCluster) sp = kMaxAttnCluster;
    // The kernel holds one CTA per SM: when the (sequence, KV head) pairs
    // times the splits exceed one wave and one wave still gives every pair
    // two splits or more, take one wave (equal-length contexts finish
    // together; a third wave of a few CTAs would cost a whole split's time)
    if (per_seq * sp > sms && sms / per_seq >= 2) sp = sms / per_seq;
  }
  // whole 128-key tiles per split (the tcgen05 kernel's tile)
  c = ((n_keys + sp - 1) / sp + 127) / 128 * 128;
  if (c < 128) c = 128;
  sp = (n_keys + c - 1) / c;
  while (!global && sp > kMaxAttnCluster) {
    c += 128;
    sp = (n_keys + c - 1) / c;
  }
  *splits = sp < 1 ? 1 : sp;
  *chunk = c;
  *merge_global = (global && *splits > 1) ? 1 : 0;
  (void)Hq;
  (void)Dh;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream, bool pdl) {
  if (a.bf16) return launch_attention_tc(a, stream, pdl);
  if (a.head_dim != 64 && a.head_dim != 128) return cudaErrorInvalidValue;
  // fp32: the per-layer slice of the caches
  const size_t layer_elems = a.page_table != nullptr
                                 ? static_cast<size_t>(a.n_pages) * a.n_kv_heads * kPageKeys * a.head_dim
                                 : static_cast<size_t>(a.max_batch) * a.n_kv_heads * a.ncap * a.head_dim;
  AttnArgs al = a;
  al.k_cache = static_cast<const float*>(a.k_cache) + layer_elems * a.layer;
  al.v_cache = static_cast<const float*>(a.v_cache) + layer_elems * a.layer;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  cfg.stream = stream;
  cfg.gridDim = dim3(a.R, a.n_q_heads, a.B);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = 0;
  return a.head_dim == 64 ? cudaLaunchKernelEx(&cfg, attn_f32_kernel<64>, al)
                          : cudaLaunchKernelEx(&cfg, attn_f32_kernel<128>, al);
}

}  // namespace dfl
