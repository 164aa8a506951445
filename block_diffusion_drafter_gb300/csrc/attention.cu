// Context attention of the drafting block over [injected context ; block]:
// every one of the R = gamma + 1 block rows of every query head attends to
// all ctx_len[b] + R keys of its KV head, with no mask (bidirectional inside
// the block; "KV Injection 메커니즘" K_i/V_i equations of "DFlash: Block
// Diffusion for Flash Speculative Decoding 논문 정리", and §3.2 of the marsggbo
// DFlash page).
//
// Memory-bound over the keys with only G*R queries per KV head (G query heads
// share one KV head), so the key range is split over CTAs (split-KV): each
// CTA streams its slice of K and V once with 16-byte cp.async loads into a
// 3-stage swizzled shared-memory ring, computes S = Q K^T and O = P V on the
// tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate) with an online
// softmax kept in registers (quad shuffles), and the last CTA of each
// (sequence, KV head) merges the split partials in a fixed order.
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"

namespace dfl {
namespace {

constexpr int kKeyTile = 64;
constexpr int kStagesKV = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxAttnCluster = 16;  // split-KV CTAs of one (sequence, KV head): one cluster

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Byte offset of 16-byte chunk `c` of row `r` in a swizzled [rows][DH] bf16 tile.
template <int DH>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * DH * 2 + ((c ^ (r & 7)) << 4));
}

// Split-partial layout: O (unnormalised, fp32) [cta][qr_pad][DH] and (m, l)
// [cta][qr_pad] (m in the log2 domain), cta = (b*Hkv + kvh)*splits + s.
template <int DH>
__global__ void __launch_bounds__(256) attn_bf16_kernel(const AttnArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int nw = blockDim.x >> 5;
  const int qr_pad = nw * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = p.n_q_heads / p.n_kv_heads;
  const int n_q = G * p.R;
  const int tile_bytes = kKeyTile * DH * 2;
  uint8_t* q_s = smem;
  uint8_t* k_s = smem + qr_pad * DH * 2;
  uint8_t* v_s = k_s + kStagesKV * tile_bytes;
  const uint32_t q_u = smem_u32(q_s), k_u = smem_u32(k_s), v_u = smem_u32(v_s);

  pdl_launch_dependents();
  pdl_wait();

  const int n_keys = p.ctx_len[b] + p.R;
  const int k_begin = s * p.chunk;
  const int k_end = (s == p.splits - 1) ? n_keys : min(n_keys, (s + 1) * p.chunk);
  const size_t hq_stride = static_cast<size_t>(p.n_q_heads) * DH;
  const size_t kv_base = (static_cast<size_t>(b) * p.n_kv_heads + kvh) * p.ncap * DH;
  const __nv_bfloat16* kg = reinterpret_cast<const __nv_bfloat16*>(p.k_cache) + kv_base;
  const __nv_bfloat16* vg = reinterpret_cast<const __nv_bfloat16*>(p.v_cache) + kv_base;
  constexpr int CH = DH / 8;  // 16-byte chunks per row

  // Q rows qr = g*R + i (query head kvh*G + g, block row i); pad rows zero.
  const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(p.q);
  for (int idx = threadIdx.x; idx < qr_pad * CH; idx += blockDim.x) {
    const int qr = idx / CH, c = idx % CH;
    const uint32_t dst = q_u + swz<DH>(qr, c);
    if (qr < n_q) {
      const int g = qr / p.R, i = qr % p.R;
      const __nv_bfloat16* src = qg + (static_cast<size_t>(b) * p.R + i) * hq_stride +
                                 static_cast<size_t>(kvh * G + g) * DH + c * 8;
      cp_async16(dst, src, 16);
    } else {
      cp_async16(dst, qg, 0);
    }
  }
  cp_async_commit();

  const int n_tiles = k_end > k_begin ? (k_end - k_begin + kKeyTile - 1) / kKeyTile : 0;
  auto load_tile = [&](int t) {
    const int st = t % kStagesKV;
    const int kb = k_begin + t * kKeyTile;
    for (int idx = threadIdx.x; idx < kKeyTile * CH; idx += blockDim.x) {
      const int r = idx / CH, c = idx % CH;
      const int key = kb + r;
      const int bytes = key < k_end ? 16 : 0;
      const size_t off = static_cast<size_t>(key < k_end ? key : k_begin) * DH + c * 8;
      cp_async16(k_u + st * tile_bytes + swz<DH>(r, c), kg + off, bytes);
      cp_async16(v_u + st * tile_bytes + swz<DH>(r, c), vg + off, bytes);
    }
  };
  // the first kStagesKV - 1 tiles go out together with Q
#pragma unroll
  for (int t = 0; t < kStagesKV - 1; ++t) {
    if (t < n_tiles) load_tile(t);
    cp_async_commit();
  }

  // Q fragments of this warp's 16 rows.
  cp_async_wait<kStagesKV - 1>();
  __syncthreads();
  uint32_t qa[DH / 16][4];
  {
    const int mat = lane >> 3, r = lane & 7;
    const int row = warp * 16 + r + (mat & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < DH / 16; ++kk)
      ldsm_x4(q_u + swz<DH>(row, kk * 2 + (mat >> 1)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
  }

  float o[DH / 8][4];
#pragma unroll
  for (int i = 0; i < DH / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float scale = rsqrtf(static_cast<float>(DH)) * kLog2e;
  const int t4 = lane & 3, g8 = lane >> 2;

  for (int t = 0; t < n_tiles; ++t) {
    cp_async_wait<kStagesKV - 2>();
    __syncthreads();
    const int st = t % kStagesKV;
    const uint32_t ks = k_u + st * tile_bytes, vs = v_u + st * tile_bytes;
    const int kb = k_begin + t * kKeyTile;
    float sc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
    {
      const int mat = lane >> 3, r = lane & 7;
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(ks + swz<DH>(16 * j + r + (mat >> 1) * 8, 2 * kk + (mat & 1)), b0, b1, b2, b3);
          mma_bf16(sc[2 * j], qa[kk], b0, b1);
          mma_bf16(sc[2 * j + 1], qa[kk], b2, b3);
        }
      }
    }
    // scale, mask, online softmax (rows g8 and g8 + 8 of this warp)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      const int key = kb + nt * 8 + 2 * t4;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const bool valid = key + q < k_end;
        sc[nt][q] = valid ? sc[nt][q] * scale : -INFINITY;
        sc[nt][2 + q] = valid ? sc[nt][2 + q] * scale : -INFINITY;
        mx0 = fmaxf(mx0, sc[nt][q]);
        mx1 = fmaxf(mx1, sc[nt][2 + q]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float base0 = mn0 == -INFINITY ? 0.f : mn0, base1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = m0 == -INFINITY ? 0.f : exp2f(m0 - base0);
    const float al1 = m1 == -INFINITY ? 0.f : exp2f(m1 - base1);
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      sc[nt][0] = exp2f(sc[nt][0] - base0);
      sc[nt][1] = exp2f(sc[nt][1] - base0);
      sc[nt][2] = exp2f(sc[nt][2] - base1);
      sc[nt][3] = exp2f(sc[nt][3] - base1);
      ps0 += sc[nt][0] + sc[nt][1];
      ps1 += sc[nt][2] + sc[nt][3];
    }
    l0 = l0 * al0 + ps0;
    l1 = l1 * al1 + ps1;
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) {
      o[i][0] *= al0; o[i][1] *= al0;
      o[i][2] *= al1; o[i][3] *= al1;
    }
    {
      const int mat = lane >> 3, r = lane & 7;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t pa[4];
        pa[0] = pack_bf16(sc[2 * j][0], sc[2 * j][1]);
        pa[1] = pack_bf16(sc[2 * j][2], sc[2 * j][3]);
        pa[2] = pack_bf16(sc[2 * j + 1][0], sc[2 * j + 1][1]);
        pa[3] = pack_bf16(sc[2 * j + 1][2], sc[2 * j + 1][3]);
#pragma unroll
        for (int e2 = 0; e2 < DH / 16; ++e2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vs + swz<DH>(16 * j + r + (mat & 1) * 8, 2 * e2 + (mat >> 1)), b0, b1, b2, b3);
          mma_bf16(o[2 * e2], pa, b0, b1);
          mma_bf16(o[2 * e2 + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();
    if (t + kStagesKV - 1 < n_tiles) load_tile(t + kStagesKV - 1);
    cp_async_commit();
  }
  cp_async_wait<0>();

  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  const int qr0 = warp * 16 + g8, qr1 = qr0 + 8;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
  auto out_index = [&](int qr, int d) -> size_t {
    const int g = qr / p.R, i = qr % p.R;
    return (static_cast<size_t>(b) * p.R + i) * hq_stride + static_cast<size_t>(kvh * G + g) * DH + d;
  };
  if (p.splits == 1) {
#pragma unroll
    for (int i = 0; i < DH / 8; ++i) {
      const int d = i * 8 + 2 * t4;
      if (qr0 < n_q) {
        const float inv = l0 > 0.f ? 1.f / l0 : 0.f;
        *reinterpret_cast<__nv_bfloat162*>(&out[out_index(qr0, d)]) =
            __floats2bfloat162_rn(o[i][0] * inv, o[i][1] * inv);
      }
      if (qr1 < n_q) {
        const float inv = l1 > 0.f ? 1.f / l1 : 0.f;
        *reinterpret_cast<__nv_bfloat162*>(&out[out_index(qr1, d)]) =
            __floats2bfloat162_rn(o[i][2] * inv, o[i][3] * inv);
      }
    }
    return;
  }

  // Split-KV merge inside the cluster of this (sequence, KV head): every CTA
  // parks its unnormalised O rows and (m, l) in its own shared memory; after
  // the barrier, CTA r merges a slice of the rows by reading all splits
  // through distributed shared memory (ascending split order), weighting each
  // split by 2^(m_s - M) / L. The second barrier keeps the partials alive
  // until every peer has read them.
  __syncthreads();  // the K/V ring is drained: reuse it for the partials
  float* po_s = reinterpret_cast<float*>(k_s);                        // [qr_pad][DH]
  float2* ml_s = reinterpret_cast<float2*>(po_s + qr_pad * DH);       // [qr_pad]
  float* w_loc = reinterpret_cast<float*>(ml_s + qr_pad);             // [rows of this CTA][splits]
#pragma unroll
  for (int i = 0; i < DH / 8; ++i) {
    const int d = i * 8 + 2 * t4;
    *reinterpret_cast<float2*>(&po_s[qr0 * DH + d]) = make_float2(o[i][0], o[i][1]);
    *reinterpret_cast<float2*>(&po_s[qr1 * DH + d]) = make_float2(o[i][2], o[i][3]);
  }
  if (t4 == 0) {
    ml_s[qr0] = make_float2(m0, l0);
    ml_s[qr1] = make_float2(m1, l1);
  }
  cluster_sync();
  const int rank = static_cast<int>(cluster_ctarank());
  const int per = (n_q + p.splits - 1) / p.splits;
  const int r0 = rank * per, r1 = min(n_q, r0 + per);
  const int nrows = r1 > r0 ? r1 - r0 : 0;
  const int S = p.splits;
  const uint32_t po_u = smem_u32(po_s), ml_u = smem_u32(ml_s);
  float2* mls = reinterpret_cast<float2*>(w_loc + ((per * S + 1) & ~1));   // [row][split] (m, l)
  // (m, l) of every (row, split) pair in parallel: one DSMEM load each
  for (int pi = threadIdx.x; pi < nrows * S; pi += blockDim.x) {
    const int qr = r0 + pi / S, sp = pi % S;
    float2 ml;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];"
                 : "=f"(ml.x), "=f"(ml.y)
                 : "r"(mapa_shared(ml_u + qr * 8, sp))
                 : "memory");
    mls[pi] = ml;
  }
  __syncthreads();
  for (int r = threadIdx.x; r < nrows; r += blockDim.x) {
    float M = -INFINITY;
    for (int sp = 0; sp < S; ++sp)
      if (mls[r * S + sp].y > 0.f) M = fmaxf(M, mls[r * S + sp].x);
    float L = 0.f;
    for (int sp = 0; sp < S; ++sp) {
      const float2 ml = mls[r * S + sp];
      const float w = ml.y > 0.f ? exp2f(ml.x - M) : 0.f;
      w_loc[r * S + sp] = w;
      L += ml.y * w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int sp = 0; sp < S; ++sp) w_loc[r * S + sp] *= inv;
  }
  __syncthreads();
  // O rows: every split's float4 is requested before any is summed; the sum
  // runs in ascending split order.
  constexpr int D4 = DH / 4;
  const int n_items = nrows * D4;
  for (int it = threadIdx.x; it < n_items; it += blockDim.x) {
    const int r = it / D4, qr = r0 + r, d = (it % D4) * 4;
    const uint32_t off = po_u + static_cast<uint32_t>((qr * DH + d) * 4);
    float4 v[kMaxAttnCluster];
#pragma unroll
    for (int sp = 0; sp < kMaxAttnCluster; ++sp)
      if (sp < S) v[sp] = ld_dsmem_f4(mapa_shared(off, sp));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int sp = 0; sp < kMaxAttnCluster; ++sp) {
      if (sp < S) {
        const float w = w_loc[r * S + sp];
        acc.x += v[sp].x * w; acc.y += v[sp].y * w; acc.z += v[sp].z * w; acc.w += v[sp].w * w;
      }
    }
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(&out[out_index(qr, d)]);
    dst[0] = __floats2bfloat162_rn(acc.x, acc.y);
    dst[1] = __floats2bfloat162_rn(acc.z, acc.w);
  }
  cluster_sync();
}

}  // namespace
}  // namespace dfl

namespace dfl {
namespace {

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
  const int n_keys = p.ctx_len[b] + p.R;
  const size_t hq_stride = static_cast<size_t>(p.n_q_heads) * DH;
  const float* q = reinterpret_cast<const float*>(p.q) + (static_cast<size_t>(b) * p.R + i) * hq_stride + hq * DH;
  const size_t kv_base = (static_cast<size_t>(b) * p.n_kv_heads + kvh) * p.ncap * DH;
  const float* kg = reinterpret_cast<const float*>(p.k_cache) + kv_base;
  const float* vg = reinterpret_cast<const float*>(p.v_cache) + kv_base;
  float qv[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) qv[d] = q[d];
  const float scale = rsqrtf(static_cast<float>(DH)) * kLog2e;
  float m = -INFINITY, l = 0.f, o[DH];
#pragma unroll
  for (int d = 0; d < DH; ++d) o[d] = 0.f;
  for (int j = threadIdx.x; j < n_keys; j += blockDim.x) {
    const float* kr = kg + static_cast<size_t>(j) * DH;
    float sdot = 0.f;
#pragma unroll
    for (int d = 0; d < DH; ++d) sdot += qv[d] * kr[d];
    sdot *= scale;
    const float mn = fmaxf(m, sdot);
    const float al = m == -INFINITY ? 0.f : exp2f(m - mn);
    const float pj = exp2f(sdot - mn);
    l = l * al + pj;
    const float* vr = vg + static_cast<size_t>(j) * DH;
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

void plan_attention(int B, int R, int Hq, int Hkv, int Dh, int max_ctx, int ncap, int* splits,
                    int* chunk) {
  const int n_keys = (max_ctx < ncap ? max_ctx : ncap) + R;
  const int per_seq = B * Hkv > 0 ? B * Hkv : 1;
  int target = (2 * 152 + per_seq - 1) / per_seq;   // ~2 CTAs per SM in total
  if (target > kMaxAttnCluster) target = kMaxAttnCluster;
  int c = (n_keys + target - 1) / target;
  c = (c + kKeyTile - 1) / kKeyTile * kKeyTile;
  if (c < 128) c = 128;
  int sp = (n_keys + c - 1) / c;
  while (sp > kMaxAttnCluster) {
    c += kKeyTile;
    sp = (n_keys + c - 1) / c;
  }
  if (const char* e = getenv("DFLASH_ATTN_SPLITS")) {   // tuning override
    sp = atoi(e);
    if (sp < 1) sp = 1;
    if (sp > kMaxAttnCluster) sp = kMaxAttnCluster;
    c = ((n_keys + sp - 1) / sp + kKeyTile - 1) / kKeyTile * kKeyTile;
    sp = (n_keys + c - 1) / c;
  }
  *splits = sp < 1 ? 1 : sp;
  *chunk = c;
  (void)Hq;
  (void)Dh;
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  cfg.stream = stream;
  if (!a.bf16) {
    cfg.gridDim = dim3(a.R, a.n_q_heads, a.B);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = 0;
    if (a.head_dim == 64) return cudaLaunchKernelEx(&cfg, attn_f32_kernel<64>, a);
    if (a.head_dim == 128) return cudaLaunchKernelEx(&cfg, attn_f32_kernel<128>, a);
    return cudaErrorInvalidValue;
  }
  const int G = a.n_q_heads / a.n_kv_heads;
  const int nw = (G * a.R + 15) / 16;
  if (nw > 8) return cudaErrorInvalidValue;
  cfg.gridDim = dim3(a.splits, a.n_kv_heads, a.B);
  cfg.blockDim = dim3(nw * 32, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(nw) * 16 * a.head_dim * 2 +
                         static_cast<size_t>(kStagesKV) * 2 * kKeyTile * a.head_dim * 2;
  void (*kern)(const AttnArgs) = a.head_dim == 128 ? attn_bf16_kernel<128> : attn_bf16_kernel<64>;
  if (a.head_dim != 64 && a.head_dim != 128) return cudaErrorInvalidValue;
  static bool configured[2][64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  bool& done = configured[a.head_dim == 128][dev & 63];
  if (!done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    done = true;
  }
  if (a.splits > kMaxAttnCluster) return cudaErrorInvalidValue;
  cudaLaunchAttribute attr2[2];
  int n = 0;
  if (pdl) {
    attr2[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr2[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (a.splits > 1) {
    attr2[n].id = cudaLaunchAttributeClusterDimension;
    attr2[n].val.clusterDim.x = a.splits;
    attr2[n].val.clusterDim.y = 1;
    attr2[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = n ? attr2 : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace dfl
