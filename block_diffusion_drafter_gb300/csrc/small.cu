// Row kernels of the drafting step: block embedding, RMSNorm, the context
// fusion's normalisation pass, argmax decoding, KV-length advance and the
// greedy verify-accept. All reductions use a fixed order (deterministic).
#include "common.cuh"
#include "internal.h"

namespace dfl {
namespace {

template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern k, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, args...);
}

// Loads of one row are issued up front (float4, up to kRowVec per thread) so a
// row costs one memory latency rather than one per strided iteration.
constexpr int kRowVec = 8;  // rows up to 256 threads x 8 float4 = 8192 floats

template <typename T>
__device__ __forceinline__ void store4(T* dst, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float4 v) {
  *reinterpret_cast<float4*>(dst) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float4 v) {
  __nv_bfloat162* d = reinterpret_cast<__nv_bfloat162*>(dst);
  d[0] = __floats2bfloat162_rn(v.x, v.y);
  d[1] = __floats2bfloat162_rn(v.z, v.w);
}
template <typename T>
__device__ __forceinline__ float4 load4(const T* src);
template <>
__device__ __forceinline__ float4 load4<float>(const float* src) {
  return *reinterpret_cast<const float4*>(src);
}
template <>
__device__ __forceinline__ float4 load4<__nv_bfloat16>(const __nv_bfloat16* src) {
  const __nv_bfloat162* s = reinterpret_cast<const __nv_bfloat162*>(src);
  const float2 a = __bfloat1622float2(s[0]), b = __bfloat1622float2(s[1]);
  return make_float4(a.x, a.y, b.x, b.y);
}

// x - bf16(x) per component (the lo part of a split bf16 value); 0 for fp32.
template <typename T>
__device__ __forceinline__ float4 sub_hi4(float4 x);
template <>
__device__ __forceinline__ float4 sub_hi4<float>(float4) { return make_float4(0.f, 0.f, 0.f, 0.f); }
template <>
__device__ __forceinline__ float4 sub_hi4<__nv_bfloat16>(float4 x) {
  auto r = [](float v) { return v - __bfloat162float(__float2bfloat16_rn(v)); };
  return make_float4(r(x.x), r(x.y), r(x.z), r(x.w));
}

template <typename T>
__global__ void __launch_bounds__(256) embed_kernel(const T* embed, const int* anchor, const int* ids,
                                                    int mask_id, int R, int D, int V, float* h, const T* gain,
                                                    T* xg, size_t xg_lo_off, float* ss,
                                                    int* dev_status) {
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.x, b = r / R, i = r % R;
  // explicit block ids (multi-step drafting), else [anchor, m, ..., m]
  int id = ids != nullptr ? ids[r] : (i == 0 ? anchor[b] : mask_id);
  if (id < 0 || id >= V) {
    if (threadIdx.x == 0) report(dev_status, DFLASH_ERR_INVALID_ARG);
    id = 0;
  }
  const T* src = embed + static_cast<size_t>(id) * D;
  float* dst = h + static_cast<size_t>(r) * D;
  T* xr = xg + static_cast<size_t>(r) * D;
  const int n4 = D / 4;
  float4 v[kRowVec];
#pragma unroll
  for (int i4 = 0; i4 < kRowVec; ++i4) {
    const int q = threadIdx.x + i4 * blockDim.x;
    if (q < n4) v[i4] = load4<T>(src + 4 * q);
  }
#pragma unroll
  for (int i4 = 0; i4 < kRowVec; ++i4) {
    const int q = threadIdx.x + i4 * blockDim.x;
    if (q < n4) {
      reinterpret_cast<float4*>(dst)[q] = v[i4];
      const float4 g = load4<T>(gain + 4 * q);
      const float4 x = make_float4(g.x * v[i4].x, g.y * v[i4].y, g.z * v[i4].z, g.w * v[i4].w);
      store4<T>(xr + 4 * q, x);
      if (xg_lo_off) store4<T>(xr + xg_lo_off + 4 * q, sub_hi4<T>(x));
    }
    // one warp holds one 128-feature slot (32 lanes x 4 features): sum of h^2
    // per slot in a fixed shuffle order
    float sq = q < n4 ? v[i4].x * v[i4].x + v[i4].y * v[i4].y + v[i4].z * v[i4].z + v[i4].w * v[i4].w : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
    if ((threadIdx.x & 31) == 0 && q < n4) ss[static_cast<size_t>(r) * (D / 128) + q / 32] = sq;
  }
}

template <typename T>
__global__ void __launch_bounds__(256) fuse_norm_kernel(const float* u, T* h, const float* row_ss,
                                                        int n_ss, const T* gain, int D, float eps) {
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.x;
  const float* ur = u + static_cast<size_t>(r) * D;
  T* row = h + static_cast<size_t>(r) * D;
  const int n4 = D / 4;
  float4 v[kRowVec];
#pragma unroll
  for (int i = 0; i < kRowVec; ++i) {
    const int q = threadIdx.x + i * blockDim.x;
    v[i] = q < n4 ? reinterpret_cast<const float4*>(ur)[q] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
  for (int s = 0; s < n_ss; ++s) ss += row_ss[static_cast<size_t>(r) * n_ss + s];
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(D) + eps);
#pragma unroll
  for (int i = 0; i < kRowVec; ++i) {
    const int q = threadIdx.x + i * blockDim.x;
    if (q < n4) {
      const float4 g = load4<T>(gain + 4 * q);
      store4<T>(row + 4 * q, make_float4(g.x * v[i].x * inv, g.y * v[i].y * inv, g.z * v[i].z * inv,
                                         g.w * v[i].w * inv));
    }
  }
}

// Block size of sequence b: gamma_b[b] clamped to [1, gamma], or gamma.
__device__ __forceinline__ int block_gamma(const int32_t* gamma_b, int b, int gamma) {
  return gamma_b == nullptr ? gamma : min(max(gamma_b[b], 1), gamma);
}

// Token i's argmax over the vocabulary: the max of the LM head's per-tile
// keys[i * ld + t] (t < n_tiles, contiguous per token), one CTA per token,
// every thread with all of its (up to kFinPer) loads in flight; the max of
// packed keys is order-free.
constexpr int kFinThreads = 128, kFinPer = 10;
__global__ void __launch_bounds__(kFinThreads) argmax_finalize_kernel(const unsigned long long* keys, int n_tiles,
                                                                      int ld, int n, int gamma,
                                                                      const int32_t* gamma_b, int32_t* draft) {
  __shared__ unsigned long long red[kFinThreads / 32];
  pdl_launch_dependents();
  pdl_wait();
  const int i = blockIdx.x;
  const unsigned long long* row = keys + static_cast<size_t>(i) * ld;
  unsigned long long best = 0ull;
  for (int t0 = 0; t0 < n_tiles; t0 += kFinThreads * kFinPer) {
    unsigned long long k[kFinPer];
#pragma unroll
    for (int u = 0; u < kFinPer; ++u) {
      const int t = t0 + u * kFinThreads + static_cast<int>(threadIdx.x);
      k[u] = t < n_tiles ? row[t] : 0ull;
    }
#pragma unroll
    for (int u = 0; u < kFinPer; ++u) best = k[u] > best ? k[u] : best;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long x = __shfl_xor_sync(0xffffffffu, best, o);
    best = x > best ? x : best;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 1; w < kFinThreads / 32; ++w) best = red[w] > best ? red[w] : best;
    draft[i] = i % gamma < block_gamma(gamma_b, i / gamma, gamma) ? static_cast<int32_t>(argmax_key_index(best))
                                                                   : -1;
  }
}

__global__ void kv_advance_kernel(int32_t* ctx_len, const int32_t* n_new, int B, int Tmax, int ncap,
                                  int reserve, int* dev_status) {
  pdl_launch_dependents();
  pdl_wait();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int nn = n_new[b];
  if (nn < 0 || nn > Tmax) { report(dev_status, DFLASH_ERR_INVALID_ARG); return; }
  if (ctx_len[b] + nn > ncap - reserve) { report(dev_status, DFLASH_ERR_CAPACITY); return; }
  ctx_len[b] += nn;
}

// Failure-detection self-test: one thread waits on an mbarrier that nothing
// arrives on, through the bounded wait every kernel of the library uses
// (about 1 s of SM clock), then reports DFLASH_ERR_TIMEOUT. No asynchronous
// copy or tensor-core work is in flight, so the CTA exits cleanly and the
// context stays usable.
__global__ void wait_selftest_kernel(int* dev_status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  if (!mbar_wait(smem_u32(&bar), 0)) report(dev_status, DFLASH_ERR_TIMEOUT);
}

__global__ void copy_f32_kernel(float* dst, const float* src, size_t n) {
  pdl_launch_dependents();
  pdl_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    dst[i] = src[i];
}

// Greedy verification. Grid (chunks, R, B): each CTA takes the argmax of one
// V-slice of target row (b, j) and folds it into keys[b*R + j] with a 64-bit
// integer max (ties -> lowest index); the last CTA of sequence b scans the
// R argmaxes against the draft and writes tau / committed / next anchor.
template <typename T>
__global__ void __launch_bounds__(256) verify_kernel(const T* logits, const int32_t* draft,
                                                     const int32_t* gamma_b, int gamma,
                                                     int V, int chunk, int32_t* tau,
                                                     int32_t* committed, int32_t* next_anchor,
                                                     unsigned long long* keys, int* counters) {
  __shared__ unsigned long long red[8];
  __shared__ int is_last;
  pdl_launch_dependents();
  pdl_wait();
  const int c = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int R = gamma + 1;
  const int v0 = c * chunk, v1 = min(V, v0 + chunk);
  const T* row = logits + (static_cast<size_t>(b) * R + j) * V;
  unsigned long long best = 0ull;
  constexpr int kVec = 16 / sizeof(T);
  if ((V % kVec) == 0 && (chunk % kVec) == 0) {
    // four 16-byte loads in flight per thread before any is compared: the
    // scan is latency-bound, not bandwidth-bound, at a few loads per thread
    constexpr int kIn = 4;
    const int stride = blockDim.x * kVec;
    int v = v0 + threadIdx.x * kVec;
    for (; v + (kIn - 1) * stride < v1; v += kIn * stride) {
      uint4 raw[kIn];
#pragma unroll
      for (int u = 0; u < kIn; ++u) raw[u] = __ldg(reinterpret_cast<const uint4*>(row + v + u * stride));
#pragma unroll
      for (int u = 0; u < kIn; ++u) {
        const T* e = reinterpret_cast<const T*>(&raw[u]);
#pragma unroll
        for (int q = 0; q < kVec; ++q) {
          const unsigned long long k = argmax_key(to_f32(e[q]), static_cast<uint32_t>(v + u * stride + q));
          best = k > best ? k : best;
        }
      }
    }
    for (; v < v1; v += stride) {
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(row + v));
      const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
      for (int q = 0; q < kVec; ++q) {
        const unsigned long long k = argmax_key(to_f32(e[q]), static_cast<uint32_t>(v + q));
        best = k > best ? k : best;
      }
    }
  } else {
    for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
      const unsigned long long k = argmax_key(to_f32(row[v]), static_cast<uint32_t>(v));
      best = k > best ? k : best;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(0xffffffffu, best, o);
    best = t > best ? t : best;
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned long long m = 0ull;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) m = red[w] > m ? red[w] : m;
    atomicMax(&keys[b * R + j], m);
    __threadfence();
    const int prev = atomicAdd(&counters[b], 1);
    is_last = prev == gridDim.x * R - 1;
  }
  __syncthreads();
  if (!is_last || threadIdx.x != 0) return;
  __threadfence();
  const int gb = block_gamma(gamma_b, b, gamma);  // this sequence's block size
  int a = 0;
  int32_t t_a = 0;
  for (int jj = 0; jj <= gb; ++jj) {
    const int32_t tj = static_cast<int32_t>(argmax_key_index(__ldcg(&keys[b * R + jj])));
    if (jj == a) {
      if (jj < gb && draft[b * gamma + jj] == tj) {
        committed[b * R + jj] = tj;
        ++a;
      } else {
        t_a = tj;
      }
    }
  }
  committed[b * R + a] = t_a;
  for (int jj = a + 1; jj <= gamma; ++jj) committed[b * R + jj] = -1;
  tau[b] = a + 1;
  next_anchor[b] = t_a;
  for (int jj = 0; jj <= gamma; ++jj) keys[b * R + jj] = 0ull;
  counters[b] = 0;
}

}  // namespace

cudaError_t launch_embed(const void* embed, const int* anchor, const int* ids, int mask_id, int B, int R,
                         int D, int V,
                         int bf16, float* h, const void* gain, void* xg, size_t xg_lo_off, float* ss,
                         int* dev_status, cudaStream_t s, bool pdl) {
  if (bf16)
    return launch_ex(embed_kernel<__nv_bfloat16>, dim3(B * R), dim3(256), 0, s, pdl,
                     reinterpret_cast<const __nv_bfloat16*>(embed), anchor, ids, mask_id, R, D, V, h,
                     reinterpret_cast<const __nv_bfloat16*>(gain), reinterpret_cast<__nv_bfloat16*>(xg),
                     xg_lo_off, ss, dev_status);
  return launch_ex(embed_kernel<float>, dim3(B * R), dim3(256), 0, s, pdl,
                   reinterpret_cast<const float*>(embed), anchor, ids, mask_id, R, D, V, h,
                   reinterpret_cast<const float*>(gain), reinterpret_cast<float*>(xg), size_t(0), ss,
                   dev_status);
}

cudaError_t launch_fuse_norm(const float* u, void* h, const float* row_ss, int n_ss, const void* gain,
                             int T, int D, float eps, int bf16, cudaStream_t s, bool pdl) {
  if (bf16)
    return launch_ex(fuse_norm_kernel<__nv_bfloat16>, dim3(T), dim3(256), 0, s, pdl, u,
                     reinterpret_cast<__nv_bfloat16*>(h), row_ss, n_ss,
                     reinterpret_cast<const __nv_bfloat16*>(gain), D, eps);
  return launch_ex(fuse_norm_kernel<float>, dim3(T), dim3(256), 0, s, pdl, u, reinterpret_cast<float*>(h),
                   row_ss, n_ss, reinterpret_cast<const float*>(gain), D, eps);
}

cudaError_t launch_argmax_finalize(const unsigned long long* keys, int n_tiles, int ld, int n, int gamma,
                                   const int32_t* gamma_b, int32_t* draft, cudaStream_t s, bool pdl) {
  return launch_ex(argmax_finalize_kernel, dim3(n), dim3(kFinThreads), 0, s, pdl, keys, n_tiles, ld, n, gamma,
                   gamma_b, draft);
}

cudaError_t launch_kv_advance(int32_t* ctx_len, const int32_t* n_new, int B, int Tmax, int ncap,
                              int reserve, int* dev_status, cudaStream_t s, bool pdl) {
  return launch_ex(kv_advance_kernel, dim3((B + 127) / 128), dim3(128), 0, s, pdl, ctx_len, n_new, B,
                   Tmax, ncap, reserve, dev_status);
}

cudaError_t launch_wait_selftest(int* dev_status, cudaStream_t s) {
  return launch_ex(wait_selftest_kernel, dim3(1), dim3(32), 0, s, false, dev_status);
}

cudaError_t launch_copy_f32(float* dst, const float* src, size_t n, cudaStream_t s, bool pdl) {
  return launch_ex(copy_f32_kernel, dim3(304), dim3(256), 0, s, pdl, dst, src, n);
}

int verify_chunks(int B, int R, int V, int num_sms) {
  int by_size = (V + 4095) / 4096;
  int by_grid = (2 * (num_sms > 0 ? num_sms : 1) + B * R - 1) / (B * R);
  int c = by_size < by_grid ? by_size : by_grid;
  return c < 1 ? 1 : c;
}

cudaError_t launch_verify(const void* logits, int bf16, const int32_t* draft, const int32_t* gamma_b,
                          int B, int gamma, int V, int32_t* tau, int32_t* committed,
                          int32_t* next_anchor, unsigned long long* keys, int* counters,
                          cudaStream_t s, bool pdl) {
  const int R = gamma + 1;
  const int chunks = verify_chunks(B, R, V, num_sms_of_current_device());
  int chunk = (V + chunks - 1) / chunks;
  chunk = (chunk + 7) / 8 * 8;
  const int n_chunks = (V + chunk - 1) / chunk;
  if (bf16)
    return launch_ex(verify_kernel<__nv_bfloat16>, dim3(n_chunks, R, B), dim3(256), 0, s, pdl,
                     reinterpret_cast<const __nv_bfloat16*>(logits), draft, gamma_b, gamma, V, chunk,
                     tau, committed, next_anchor, keys, counters);
  return launch_ex(verify_kernel<float>, dim3(n_chunks, R, B), dim3(256), 0, s, pdl,
                   reinterpret_cast<const float*>(logits), draft, gamma_b, gamma, V, chunk, tau,
                   committed, next_anchor, keys, counters);
}

int num_sms_of_current_device() {
  // SM count of each device, queried once (0: not yet known). A failed query
  // gives 1: plans stay valid, only the grid sizing is poorer, and the launch
  // that follows reports the device error itself.
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  int& n = cached[dev & 63];
  if (n == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) return 1;
    n = v;
  }
  return n;
}

}  // namespace dfl
