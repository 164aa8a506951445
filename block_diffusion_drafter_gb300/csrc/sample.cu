// Sampling verification (temperature > 0) of a drafted block: the
// rejection-acceptance rule that keeps speculative decoding lossless in
// distribution ("DFlash 블록 확산 디코딩" lossless paragraph; "DFlash: Block
// Diffusion for Flash Speculative Decoding 논문 정리" temperature-1 results):
//   p_j = softmax(target_j / T), q_j = softmax(draft_logits_j / T);
//   draft j is kept while u_j * q_j(x_j) < p_j(x_j), u_j ~ U(0, 1);
//   at the first rejection a the replacement is a draw from
//   norm(max(p_a - q_a, 0)) (from p_a if that has no mass); after gamma
//   kept drafts the bonus is a draw from p_gamma.
// Draws are Gumbel-max over V with splitmix64 noise (common.cuh).
//
// Three launches over one workspace region:
//   1. sample_stats_kernel: grid (V chunks, B x (2 gamma + 1) rows): per row
//      and chunk the max m of logit / T and sum exp(logit / T - m);
//   2. sample_decide_kernel: one CTA per sequence merges each row's chunks
//      (a warp per row, fixed tree) and scans the acceptance test;
//   3. sample_resid_kernel: grid (512-entry V chunks, B): per chunk the best packed
//      (score, index) key of the residual and of the plain p_a / p_gamma
//      draw, atomicMax per sequence; the last CTA of a sequence decides.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dfl {
namespace {

constexpr int kStatThreads = 256;
constexpr int kPerThread = kSampChunk / kStatThreads;
constexpr int kMaxGammaSample = 32;  // block rows the decision kernel holds (gamma <= 16)
constexpr int kResidChunk = 512;     // vocabulary entries per residual-draw CTA
constexpr int kResidPer = kResidChunk / kStatThreads;

template <typename T>
__device__ __forceinline__ float logit_at(const T* p, size_t i);
template <>
__device__ __forceinline__ float logit_at<float>(const float* p, size_t i) { return p[i]; }
template <>
__device__ __forceinline__ float logit_at<__nv_bfloat16>(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}

// Block-wide reductions in a fixed tree over 256 threads.
__device__ __forceinline__ float block_max256(float v, float* red) {
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
__device__ __forceinline__ float block_sum256(float v, float* red) {
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
__device__ __forceinline__ unsigned long long block_keymax256(unsigned long long v,
                                                              unsigned long long* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long u = __shfl_xor_sync(0xffffffffu, v, o);
    v = u > v ? u : v;
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  unsigned long long t = lane < 8 ? red[lane] : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long u = __shfl_xor_sync(0xffffffffu, t, o);
    t = u > t ? u : t;
  }
  return t;
}

// Row r of sequence b: r <= gamma a target row, r > gamma draft row r - gamma - 1.
template <typename TT>
__global__ void __launch_bounds__(kStatThreads)
    sample_stats_kernel(const TT* target, const float* draft_logits, int gamma, int V, float inv_t,
                        int n_chunks, float2* partials) {
  __shared__ float red[8];
  pdl_launch_dependents();
  pdl_wait();
  const int c = blockIdx.x, row = blockIdx.y;
  const int R = gamma + 1, nrow = 2 * gamma + 1;
  const int b = row / nrow, r = row % nrow;
  float x[kPerThread];
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kPerThread; ++i) {
    const int v = c * kSampChunk + threadIdx.x + i * kStatThreads;
    x[i] = -INFINITY;
    if (v < V)
      x[i] = (r < R ? logit_at(target, (static_cast<size_t>(b) * R + r) * V + v)
                    : draft_logits[(static_cast<size_t>(b) * gamma + (r - R)) * V + v]) * inv_t;
    m = fmaxf(m, x[i]);
  }
  m = block_max256(m, red);
  float s = 0.f;
  if (m > -INFINITY) {
#pragma unroll
    for (int i = 0; i < kPerThread; ++i)
      if (x[i] > -INFINITY) s += expf(x[i] - m);
  }
  s = block_sum256(s, red);
  if (threadIdx.x == 0) partials[static_cast<size_t>(row) * n_chunks + c] = make_float2(m, s);
}

// (m, s) pairs of max and sum exp(x - m): the pair of the union.
__device__ __forceinline__ void softmax_merge(float& m, float& s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  const float nm = fmaxf(m, m2);
  s = s * expf(m - nm) + s2 * expf(m2 - nm);
  m = nm;
}

// One CTA per sequence: a warp per row merges the row's chunk statistics
// (lane-strided, then a fixed shuffle tree); the gamma candidates' p and q
// and uniforms are computed in parallel; one thread scans the acceptance
// test over shared memory.
template <typename TT>
__global__ void __launch_bounds__(1024)
    sample_decide_kernel(const TT* target, const float* draft_logits, const int32_t* draft, int gamma,
                         int V, float inv_t, uint64_t seed, int n_chunks, const float2* partials,
                         SampleState* state, unsigned long long* keys, unsigned int* counters) {
  __shared__ float mx[2 * kMaxGammaSample + 1], sm[2 * kMaxGammaSample + 1];
  __shared__ float pj[kMaxGammaSample], qj[kMaxGammaSample], uj[kMaxGammaSample];
  __shared__ int okj[kMaxGammaSample];
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x, R = gamma + 1, nrow = 2 * gamma + 1;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int r = w; r < nrow; r += blockDim.x >> 5) {
    const float2* pp = partials + (static_cast<size_t>(b) * nrow + r) * n_chunks;
    float m = -INFINITY, s = 0.f;
    for (int c = lane; c < n_chunks; c += 32) softmax_merge(m, s, pp[c].x, pp[c].y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
      // both lanes of a pair merge in the same (lower lane first) order
      if (lane & o) { float tm = m, ts = s; m = m2; s = s2; softmax_merge(m, s, tm, ts); }
      else softmax_merge(m, s, m2, s2);
    }
    if (lane == 0) { mx[r] = m; sm[r] = s; }
  }
  __syncthreads();
  const int j = threadIdx.x;
  if (j < gamma) {
    const int x = draft[static_cast<size_t>(b) * gamma + j];
    const bool ok = x >= 0 && x < V;  // not a token: rejected
    okj[j] = ok;
    pj[j] = ok ? expf(logit_at(target, (static_cast<size_t>(b) * R + j) * V + x) * inv_t - mx[j]) / sm[j] : 0.f;
    qj[j] = ok ? expf(draft_logits[(static_cast<size_t>(b) * gamma + j) * V + x] * inv_t - mx[R + j]) / sm[R + j]
               : 1.f;
    uj[j] = rng_uniform(seed, rng_counter(kStreamAccept, j, b, 0));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int a = 0;
    while (a < gamma && okj[a] && uj[a] * qj[a] < pj[a]) ++a;
    SampleState st{};
    st.a = a;
    st.mt = mx[a];
    st.st = sm[a];
    st.md = a < gamma ? mx[R + a] : 0.f;
    st.sd = a < gamma ? sm[R + a] : 1.f;
    state[b] = st;
    keys[2 * b] = 0ull;
    keys[2 * b + 1] = 0ull;
    counters[b] = 0u;
  }
}

template <typename TT>
__global__ void __launch_bounds__(kStatThreads)
    sample_resid_kernel(const TT* target, const float* draft_logits, const int32_t* draft, int gamma,
                        int V, float inv_t, uint64_t seed, int n_chunks, const SampleState* state,
                        unsigned long long* keys, unsigned int* counters, int32_t* tau,
                        int32_t* committed, int32_t* next_anchor) {
  __shared__ unsigned long long red[8];
  __shared__ bool last;
  pdl_launch_dependents();
  pdl_wait();
  const int c = blockIdx.x, b = blockIdx.y, R = gamma + 1;
  const SampleState st = state[b];
  const int a = st.a;
  const size_t trow = (static_cast<size_t>(b) * R + a) * V;
  const size_t drow = (static_cast<size_t>(b) * gamma + (a < gamma ? a : 0)) * V;
  unsigned long long best_r = 0ull, best_f = 0ull;  // residual draw, plain draw
#pragma unroll 4
  for (int i = 0; i < kResidPer; ++i) {
    const int v = c * kResidChunk + threadIdx.x + i * kStatThreads;
    if (v >= V) break;
    const float tv = logit_at(target, trow + v) * inv_t;
    if (a < gamma) {
      const float g = rng_gumbel(seed, rng_counter(kStreamResid, a, b, static_cast<uint32_t>(v)));
      const float w = expf(tv - st.mt) / st.st - expf(draft_logits[drow + v] * inv_t - st.md) / st.sd;
      if (w > 0.f) {
        const unsigned long long k = argmax_key(logf(w) + g, static_cast<uint32_t>(v));
        best_r = k > best_r ? k : best_r;
      }
      const unsigned long long k = argmax_key(tv + g, static_cast<uint32_t>(v));
      best_f = k > best_f ? k : best_f;
    } else {
      const float g = rng_gumbel(seed, rng_counter(kStreamBonus, gamma, b, static_cast<uint32_t>(v)));
      const unsigned long long k = argmax_key(tv + g, static_cast<uint32_t>(v));
      best_f = k > best_f ? k : best_f;
    }
  }
  best_r = block_keymax256(best_r, red);
  best_f = block_keymax256(best_f, red);
  if (threadIdx.x == 0) {
    if (best_r != 0ull) atomicMax(&keys[2 * b], best_r);
    if (best_f != 0ull) atomicMax(&keys[2 * b + 1], best_f);
    __threadfence();
    last = atomicAdd(&counters[b], 1u) == static_cast<unsigned int>(n_chunks - 1);
  }
  __syncthreads();
  if (!last || threadIdx.x != 0) return;
  __threadfence();
  const unsigned long long kr = *reinterpret_cast<volatile unsigned long long*>(&keys[2 * b]);
  const unsigned long long kf = *reinterpret_cast<volatile unsigned long long*>(&keys[2 * b + 1]);
  const int y = static_cast<int>(argmax_key_index(kr != 0ull ? kr : kf));
  tau[b] = a + 1;
  for (int k = 0; k < R; ++k)
    committed[static_cast<size_t>(b) * R + k] =
        k < a ? draft[static_cast<size_t>(b) * gamma + k] : (k == a ? y : -1);
  next_anchor[b] = y;
}

template <typename K, typename... Args>
cudaError_t launch_ex(K kernel, dim3 grid, dim3 block, cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct SampleLayout {
  size_t partials, state, keys, counters, total;
};
SampleLayout sample_layout(int max_batch, int gamma, int vocab) {
  const size_t n_chunks = (static_cast<size_t>(vocab) + kSampChunk - 1) / kSampChunk;
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  SampleLayout L{};
  L.partials = 0;
  L.state = up(static_cast<size_t>(max_batch) * (2 * gamma + 1) * n_chunks * sizeof(float2));
  L.keys = L.state + up(static_cast<size_t>(max_batch) * sizeof(SampleState));
  L.counters = L.keys + up(static_cast<size_t>(max_batch) * 2 * sizeof(unsigned long long));
  L.total = L.counters + up(static_cast<size_t>(max_batch) * sizeof(unsigned int));
  return L;
}

template <typename TT>
cudaError_t launch_all(const TT* target, const float* draft_logits, const int32_t* draft, int B, int gamma,
                       int V, float temp, uint64_t seed, void* ws, int32_t* tau, int32_t* committed,
                       int32_t* next_anchor, cudaStream_t s, bool pdl) {
  const SampleLayout L = sample_layout(B, gamma, V);
  uint8_t* base = static_cast<uint8_t*>(ws);
  float2* partials = reinterpret_cast<float2*>(base + L.partials);
  SampleState* state = reinterpret_cast<SampleState*>(base + L.state);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(base + L.keys);
  unsigned int* counters = reinterpret_cast<unsigned int*>(base + L.counters);
  const int n_chunks = (V + kSampChunk - 1) / kSampChunk;
  const int n_resid = (V + kResidChunk - 1) / kResidChunk;
  const float inv_t = 1.0f / temp;  // logits are scaled by 1/T in every kernel alike
  cudaError_t e = launch_ex(sample_stats_kernel<TT>, dim3(n_chunks, B * (2 * gamma + 1)),
                            dim3(kStatThreads), s, pdl, target, draft_logits, gamma, V, inv_t, n_chunks,
                            partials);
  if (e != cudaSuccess) return e;
  e = launch_ex(sample_decide_kernel<TT>, dim3(B), dim3(1024), s, pdl, target, draft_logits, draft, gamma, V,
                inv_t, seed, n_chunks, static_cast<const float2*>(partials), state, keys, counters);
  if (e != cudaSuccess) return e;
  return launch_ex(sample_resid_kernel<TT>, dim3(n_resid, B), dim3(kStatThreads), s, pdl, target,
                   draft_logits, draft, gamma, V, inv_t, seed, n_resid,
                   static_cast<const SampleState*>(state), keys, counters, tau, committed, next_anchor);
}

}  // namespace

size_t sample_ws_bytes(int max_batch, int gamma, int vocab) {
  return sample_layout(max_batch, gamma, vocab).total;
}

cudaError_t launch_sample_verify(const void* target, int target_bf16, const float* draft_logits,
                                 const int32_t* draft, int B, int gamma, int V, float temperature,
                                 uint64_t seed, void* ws, int32_t* tau, int32_t* committed,
                                 int32_t* next_anchor, cudaStream_t s, bool pdl) {
  if (target_bf16)
    return launch_all(static_cast<const __nv_bfloat16*>(target), draft_logits, draft, B, gamma, V, temperature,
                      seed, ws, tau, committed, next_anchor, s, pdl);
  return launch_all(static_cast<const float*>(target), draft_logits, draft, B, gamma, V, temperature, seed, ws,
                    tau, committed, next_anchor, s, pdl);
}

}  // namespace dfl
