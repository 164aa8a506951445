// Multi-step confidence unmasking within a block ("DFlash 블록 확산 디코딩"
// drafting paragraph: the block starts as [MASK] everywhere, every pass
// predicts all masked positions at once, the most confident positions are
// filled first and the passes repeat until the block is full). Readings:
// confidence = max_v softmax(logits_j) = 1 / sum_v exp(l_v - max l); pass s of
// S fills ceil(m / (S - s)) of the m masked positions; ties go to the lower
// position; filled positions keep their token as input to later passes.
//
// Launches per decision: conf_stats_kernel (grid V chunks x B*gamma rows: the
// max and sum exp of every row's chunk) and unmask_select_kernel (one CTA per
// sequence: combine each row's chunks in ascending order, pick, write ids).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dfl {
namespace {

constexpr int kThreads = 256;
constexpr int kPer = kSampChunk / kThreads;

__device__ __forceinline__ float bmax(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = lane < 8 ? red[lane] : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
  return t;
}
__device__ __forceinline__ float bsum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = lane < 8 ? red[lane] : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

__global__ void ids_init_kernel(const int32_t* anchor, int mask_id, int B, int R, int32_t* ids) {
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < B * R) ids[i] = i % R == 0 ? anchor[i / R] : mask_id;
}

__global__ void ids_to_draft_kernel(const int32_t* ids, int B, int gamma, int32_t* draft) {
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < B * gamma) draft[i] = ids[(i / gamma) * (gamma + 1) + 1 + i % gamma];
}

__global__ void __launch_bounds__(kThreads)
    conf_stats_kernel(const float* logits, int V, int n_chunks, float2* partials) {
  __shared__ float red[8];
  pdl_launch_dependents();
  pdl_wait();
  const int c = blockIdx.x, row = blockIdx.y;
  const float* lr = logits + static_cast<size_t>(row) * V;
  float x[kPer];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int v = c * kSampChunk + threadIdx.x + i * kThreads;
    x[i] = v < V ? lr[v] : -INFINITY;
    m = fmaxf(m, x[i]);
  }
  m = bmax(m, red);
  float s = 0.f;
  if (m > -INFINITY) {
#pragma unroll
    for (int i = 0; i < kPer; ++i)
      if (x[i] > -INFINITY) s += expf(x[i] - m);
  }
  s = bsum(s, red);
  if (threadIdx.x == 0) partials[static_cast<size_t>(row) * n_chunks + c] = make_float2(m, s);
}

__global__ void __launch_bounds__(32)
    unmask_select_kernel(const int32_t* draft, int gamma, int mask_id, int steps_left, int n_chunks,
                         const float2* partials, int32_t* ids) {
  __shared__ float conf[32];
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x, R = gamma + 1;
  const int j = threadIdx.x;
  if (j < gamma) {  // combine the row's chunks in ascending order
    const float2* pp = partials + (static_cast<size_t>(b) * gamma + j) * n_chunks;
    float m = -INFINITY;
    for (int c = 0; c < n_chunks; ++c) m = fmaxf(m, pp[c].x);
    float s = 0.f;
    for (int c = 0; c < n_chunks; ++c)
      if (pp[c].y > 0.f) s += pp[c].y * expf(pp[c].x - m);
    conf[j] = s > 0.f ? 1.f / s : 0.f;
  }
  __syncwarp();
  if (threadIdx.x != 0) return;
  int32_t* row = ids + static_cast<size_t>(b) * R + 1;
  uint32_t masked = 0u;
  int m = 0;
  for (int i = 0; i < gamma; ++i)
    if (row[i] == mask_id) { masked |= 1u << i; ++m; }
  const int k = (m + steps_left - 1) / steps_left;
  for (int t = 0; t < k; ++t) {
    int best = -1;
    for (int i = 0; i < gamma; ++i)  // most confident, lowest position on ties
      if ((masked >> i) & 1u)
        if (best < 0 || conf[i] > conf[best]) best = i;
    masked &= ~(1u << best);
    row[best] = draft[static_cast<size_t>(b) * gamma + best];
  }
}

template <typename K, typename... Args>
cudaError_t launch_ex(K kernel, dim3 grid, dim3 block, cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

cudaError_t launch_ids_init(const int32_t* anchor, int mask_id, int B, int R, int32_t* ids, cudaStream_t s,
                            bool pdl) {
  return launch_ex(ids_init_kernel, dim3((B * R + 127) / 128), dim3(128), s, pdl, anchor, mask_id, B, R, ids);
}

cudaError_t launch_ids_to_draft(const int32_t* ids, int B, int gamma, int32_t* draft, cudaStream_t s,
                                bool pdl) {
  return launch_ex(ids_to_draft_kernel, dim3((B * gamma + 127) / 128), dim3(128), s, pdl, ids, B, gamma, draft);
}

cudaError_t launch_unmask_step(const float* logits, const int32_t* draft, int B, int gamma, int V,
                               int mask_id, int steps_left, void* ws, int32_t* ids, cudaStream_t s,
                               bool pdl) {
  const int n_chunks = (V + kSampChunk - 1) / kSampChunk;
  float2* partials = static_cast<float2*>(ws);
  cudaError_t e = launch_ex(conf_stats_kernel, dim3(n_chunks, B * gamma), dim3(kThreads), s, pdl, logits, V,
                            n_chunks, partials);
  if (e != cudaSuccess) return e;
  return launch_ex(unmask_select_kernel, dim3(B), dim3(32), s, pdl, draft, gamma, mask_id, steps_left, n_chunks,
                   static_cast<const float2*>(partials), ids);
}

}  // namespace dfl
