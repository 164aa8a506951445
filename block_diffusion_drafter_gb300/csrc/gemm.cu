// Projection GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by
// TMA through an mbarrier pipeline, with the drafting step's epilogues fused.
//
// Computes C[a, b] = sum_k A[a, k] * B[b, k] for K-major (row-major [rows, k])
// A and B. One CTA owns a 128-row A tile x bn-row B tile and a contiguous
// range of k-tiles (split-K); warp 0 issues TMA, warp 1 owns TMEM and issues
// the MMAs, warps 2-5 run the epilogue. Both GEMM orientations of the step use
// it:
//  - "swap" (A = weight rows, B = tokens): the skinny decode projections,
//    where a block has only B*(gamma+1) rows; every weight byte is streamed
//    from HBM exactly once and the token tile rides along as the MMA's N.
//  - plain (A = tokens, B = weight rows): context fusion / injection over
//    long prefills, which is tensor-bound.
// Split-K partial tiles are reduced by the last-arriving CTA of a tile in a
// fixed split order (deterministic; no float atomics, no inter-CTA waits).
#include <stdio.h>

#include "common.cuh"
#include "internal.h"

#include <cudaTypedefs.h>

namespace dfl {

namespace {

constexpr int kSLD = 129;  // staging row stride (floats): conflict-free both ways

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ void store_out(void* out, int bf16, size_t idx, float v) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(out)[idx] = v;
}

// Rotate-half RoPE of element d of a head given its partner value.
__device__ __forceinline__ float rope_rot(const Epi& e, int pos, int d, float x, float xp) {
  if (e.rope_cos == nullptr) return x;
  const int half = e.head_dim >> 1;
  const int j = d < half ? d : d - half;
  const size_t t = static_cast<size_t>(pos) * half + j;
  const float c = e.rope_cos[t], s = e.rope_sin[t];
  return d < half ? x * c - xp * s : x * c + xp * s;
}

// Applies the epilogue to one staged chunk: S[b * kSLD + a] holds C for
// A-row a (0..127) and B-row col0 + b (0 <= b < cols) of tile (m_tile, n_tile).
// Runs on the 128 epilogue threads (etid 0..127).
__device__ void apply_epilogue(const GemmArgs& g, const float* S, int col0, int cols, int m_tile,
                               int n_tile, int etid) {
  const Epi& e = g.epi;
  const int total = cols * kBM;
  switch (e.op) {
    case EPI_STORE:
    case EPI_ADD_F32:
    case EPI_FUSE: {
      for (int idx = etid; idx < total; idx += 128) {
        int a, b;
        if (g.swap) { a = idx & 127; b = idx >> 7; } else { b = idx % cols; a = idx / cols; }
        const int feat = g.swap ? m_tile * kBM + a : n_tile * g.bn + col0 + b;
        const int tok = g.swap ? n_tile * g.bn + col0 + b : m_tile * kBM + a;
        if (tok >= e.n_tok || feat >= e.n_feat) continue;
        const float v = S[b * kSLD + a];
        const size_t o = static_cast<size_t>(tok) * e.ld + feat;
        if (e.op == EPI_ADD_F32)
          reinterpret_cast<float*>(e.out)[o] += v;
        else
          store_out(e.out, e.out_bf16, o, v);
      }
      if (e.op == EPI_FUSE) {
        // Per token: sum of squares over this chunk's 128 features, summed
        // sequentially (fixed order), one slot per 128-feature group.
        if (g.swap) {
          const int b = etid;
          const int tok = n_tile * g.bn + col0 + b;
          if (b < cols && tok < e.n_tok) {
            float ss = 0.f;
            for (int a = 0; a < kBM; ++a) { const float v = S[b * kSLD + a]; ss += v * v; }
            e.row_ss[static_cast<size_t>(tok) * e.n_ss + m_tile] = ss;
          }
        } else {
          const int a = etid;
          const int tok = m_tile * kBM + a;
          if (tok < e.n_tok) {
            float ss = 0.f;
            for (int b = 0; b < cols; ++b) { const float v = S[b * kSLD + a]; ss += v * v; }
            e.row_ss[static_cast<size_t>(tok) * e.n_ss + (n_tile * g.bn + col0) / kBM] = ss;
          }
        }
      }
      break;
    }
    case EPI_SWIGLU: {
      // A rows 0..63: gate features m_tile*64 + a; rows 64..127: matching up rows.
      for (int idx = etid; idx < cols * 64; idx += 128) {
        const int a = idx & 63, b = idx >> 6;
        const int feat = m_tile * 64 + a;
        const int tok = n_tile * g.bn + col0 + b;
        if (tok >= e.n_tok || feat >= e.n_feat) continue;
        const float gate = S[b * kSLD + a], up = S[b * kSLD + a + 64];
        store_out(e.out, e.out_bf16, static_cast<size_t>(tok) * e.ld + feat, silu_f(gate) * up);
      }
      break;
    }
    case EPI_QKV: {
      // swap orientation: A rows are features of the stacked [Q; K; V] projection.
      const int Dh = e.head_dim, half = Dh >> 1;
      const int nq = e.n_q_heads * Dh, nk = e.n_kv_heads * Dh;
      for (int idx = etid; idx < total; idx += 128) {
        const int a = idx & 127, b = idx >> 7;
        const int f = m_tile * kBM + a;
        const int t = n_tile * g.bn + col0 + b;
        if (t >= e.n_tok || f >= e.n_feat) continue;
        const int seq = t / e.rows_per_seq, i = t - seq * e.rows_per_seq;
        const int pos = e.ctx_len[seq] + i;
        const int d = f % Dh;
        const float x = S[b * kSLD + a];
        if (f < nq) {
          const float xp = S[b * kSLD + (d < half ? a + half : a - half)];
          store_out(e.out, e.out_bf16, static_cast<size_t>(t) * e.ld + f, rope_rot(e, pos, d, x, xp));
        } else {
          if (pos >= e.ncap) { report(g.dev_status, DFLASH_ERR_CAPACITY); continue; }
          const bool is_k = f < nq + nk;
          const int head = ((is_k ? f - nq : f - nq - nk)) / Dh;
          float y = x;
          if (is_k) y = rope_rot(e, pos, d, x, S[b * kSLD + (d < half ? a + half : a - half)]);
          const size_t o =
              ((static_cast<size_t>(e.layer) * e.max_batch + seq) * e.n_kv_heads + head) * e.ncap + pos;
          store_out(is_k ? e.k_cache : e.v_cache, e.out_bf16, o * Dh + d, y);
        }
      }
      break;
    }
    case EPI_KV: {
      const int Dh = e.head_dim, half = Dh >> 1;
      const int nk = e.n_kv_heads * Dh;
      for (int idx = etid; idx < total; idx += 128) {
        int a, b;
        if (g.swap) { a = idx & 127; b = idx >> 7; } else { b = idx % cols; a = idx / cols; }
        const int gf = g.swap ? m_tile * kBM + a : n_tile * g.bn + col0 + b;
        const int r = g.swap ? n_tile * g.bn + col0 + b : m_tile * kBM + a;
        if (r >= e.n_tok || gf >= e.n_feat) continue;
        const int seq = r / e.rows_per_seq, t = r - seq * e.rows_per_seq;
        const int nn = e.n_new[seq], base = e.ctx_len[seq];
        if (t >= nn || base + nn > e.ncap - e.reserve) continue;
        const int layer = gf / e.feat_per_layer, f = gf - layer * e.feat_per_layer;
        const bool is_k = f < nk;
        const int fk = is_k ? f : f - nk;
        const int head = fk / Dh, d = fk % Dh;
        const int pos = base + t;
        const float x = S[b * kSLD + a];
        float y = x;
        if (is_k) {
          const int pa = g.swap ? (d < half ? a + half : a - half) : a;
          const int pb = g.swap ? b : (d < half ? b + half : b - half);
          y = rope_rot(e, pos, d, x, S[pb * kSLD + pa]);
        }
        const size_t o = ((static_cast<size_t>(layer) * e.max_batch + seq) * e.n_kv_heads + head) * e.ncap + pos;
        store_out(is_k ? e.k_cache : e.v_cache, e.out_bf16, o * Dh + d, y);
      }
      break;
    }
    case EPI_ARGMAX: {
      // swap orientation: A rows are vocabulary entries, B rows tokens.
      const int w = etid >> 5, lane = etid & 31;
      for (int b = w; b < cols; b += 4) {
        const int tok = n_tile * g.bn + col0 + b;
        unsigned long long best = 0ull;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int a = lane + 32 * i;
          const int feat = m_tile * kBM + a;
          if (feat < e.n_feat) {
            const float v = S[b * kSLD + a];
            const unsigned long long key = argmax_key(v, static_cast<uint32_t>(feat));
            best = key > best ? key : best;
            if (e.out != nullptr && tok < e.n_tok)
              reinterpret_cast<float*>(e.out)[static_cast<size_t>(tok) * e.ld + feat] = v;
          }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, off);
          best = o > best ? o : best;
        }
        if (lane == 0 && tok < e.n_tok && best != 0ull) atomicMax(&e.keys[tok], best);
      }
      break;
    }
    default:
      break;
  }
}

}  // namespace
}  // namespace dfl

namespace dfl {
namespace {

struct SmemHeader {
  uint64_t full[16];
  uint64_t empty[16];
  uint64_t accum;
  uint32_t tmem_base;
  int abort_flag;
  int last_flag;
  int epi_ok;
};

template <bool kTF32>
__global__ void __launch_bounds__(kGemmThreads)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap a_map,
                   const __grid_constant__ CUtensorMap b_map, const GemmArgs g, int stages) {
  extern __shared__ uint8_t smem_raw[];
  SmemHeader* hdr = reinterpret_cast<SmemHeader*>(smem_raw);
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t tiles_s = (raw_s + sizeof(SmemHeader) + 1023u) & ~1023u;
  uint8_t* tiles = smem_raw + (tiles_s - raw_s);

  constexpr int kBK = kTF32 ? 32 : 64;  // 128 bytes of k per row either way
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x, split = blockIdx.y, n_tile = blockIdx.z;
  const int KT = g.k / kBK;
  const int kt0 = split * g.kt_per_split;
  const int nkt = min(g.kt_per_split, KT - kt0);
  const uint32_t a_bytes = kBM * 128u;
  const uint32_t b_bytes = static_cast<uint32_t>(g.bn) * 128u;
  const uint32_t stage_bytes = a_bytes + b_bytes;
  const int sub_rows = g.bn / g.n_sub;
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(g.bn)) tmem_cols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&hdr->full[s]), 1);
      mbar_init(smem_u32(&hdr->empty[s]), 1);
    }
    mbar_init(smem_u32(&hdr->accum), 1);
    hdr->abort_flag = 0;
    hdr->last_flag = 0;
    fence_mbar_init();
    fence_proxy_async();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&hdr->tmem_base), tmem_cols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&a_map);
    tma_prefetch_map(&b_map);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol_w = l2_evict_first();
      const uint64_t pol_x = l2_evict_last();
      const uint64_t pol_a = g.a_weights ? pol_w : pol_x;
      const uint64_t pol_b = g.a_weights ? pol_x : pol_w;
      const int a_rows_per_tile = g.a_gateup > 0 ? 64 : kBM;
      const int a_y = g.a_row0 + (m_tile % g.a_tiles_per_z) * a_rows_per_tile;
      const int a_z = g.a_z0 + m_tile / g.a_tiles_per_z;
      const int b_y = g.b_row0 + (n_tile % g.b_tiles_per_z) * g.bn;
      const int b_z = g.b_z0 + n_tile / g.b_tiles_per_z;
      auto load_a = [&](int s, int kt) {
        const uint32_t dst = tiles_s + s * stage_bytes;
        const uint32_t bar = smem_u32(&hdr->full[s]);
        if (g.a_gateup > 0) {
          tma_load_3d(dst, &a_map, bar, kt * kBK, a_y, a_z, pol_a);
          tma_load_3d(dst + 64 * 128, &a_map, bar, kt * kBK, a_y + g.a_gateup, a_z, pol_a);
        } else {
          tma_load_3d(dst, &a_map, bar, kt * kBK, a_y, a_z, pol_a);
        }
      };
      auto load_b = [&](int s, int kt) {
        const uint32_t dst = tiles_s + s * stage_bytes + a_bytes;
        const uint32_t bar = smem_u32(&hdr->full[s]);
        for (int sub = 0; sub < g.n_sub; ++sub)
          tma_load_3d(dst + sub * sub_rows * 128, &b_map, bar, kt * kBK, b_y + sub * sub_rows, b_z,
                      pol_b);
      };
      // Weights do not depend on the previous kernel: start streaming them
      // before waiting for it (programmatic dependent launch).
      int n_pre = 0;
      if (g.a_weights) {
        n_pre = min(stages, nkt);
        for (int it = 0; it < n_pre; ++it) {
          mbar_expect_tx(smem_u32(&hdr->full[it]), stage_bytes);
          load_a(it, kt0 + it);
        }
      }
      pdl_wait();
      for (int it = 0; it < n_pre; ++it) load_b(it, kt0 + it);
      for (int it = n_pre; it < nkt; ++it) {
        const int s = it % stages, u = it / stages;
        if (u > 0 && !mbar_wait(smem_u32(&hdr->empty[s]), (u - 1) & 1)) {
          report(g.dev_status, DFLASH_ERR_TIMEOUT);
          atomicExch(&hdr->abort_flag, 1);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&hdr->abort_flag)) break;
        mbar_expect_tx(smem_u32(&hdr->full[s]), stage_bytes);
        load_a(s, kt0 + it);
        load_b(s, kt0 + it);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc(kBM, sub_rows, kTF32 ? kFmtTF32 : kFmtBF16);
      for (int it = 0; it < nkt; ++it) {
        const int s = it % stages, u = it / stages;
        if (!mbar_wait(smem_u32(&hdr->full[s]), u & 1)) {
          report(g.dev_status, DFLASH_ERR_TIMEOUT);
          atomicExch(&hdr->abort_flag, 1);
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = tiles_s + s * stage_bytes;
        const uint32_t b_addr = a_addr + a_bytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // 4 x 32 bytes of k per 128-byte row
          const uint64_t adesc = sw128_desc(a_addr + k * 32);
          for (int sub = 0; sub < g.n_sub; ++sub) {
            const uint64_t bdesc = sw128_desc(b_addr + sub * sub_rows * 128 + k * 32);
            const uint32_t acc = (it > 0 || k > 0) ? 1u : 0u;
            if (kTF32)
              tc_mma_tf32(tmem + sub * sub_rows, adesc, bdesc, idesc, acc);
            else
              tc_mma_f16(tmem + sub * sub_rows, adesc, bdesc, idesc, acc);
          }
        }
        tc_commit(smem_u32(&hdr->empty[s]));
      }
      tc_commit(smem_u32(&hdr->accum));
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;        // A row of this thread
    const int etid = threadIdx.x - 64;          // 0..127
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float* S = reinterpret_cast<float*>(tiles); // staging reuses the drained pipeline
    pdl_wait();
    if (!mbar_wait(smem_u32(&hdr->accum), 0)) {
      report(g.dev_status, DFLASH_ERR_TIMEOUT);
      atomicExch(&hdr->abort_flag, 1);
    }
    tc_fence_after();
    // One thread decides for all 128 so that every epilogue thread takes the
    // same path through the named barriers below.
    named_bar(1, 128);
    if (etid == 0) hdr->epi_ok = *reinterpret_cast<volatile int*>(&hdr->abort_flag) == 0 ? 1 : 0;
    named_bar(1, 128);
    const bool ok = hdr->epi_ok != 0;
    if (ok) {
      const int n_chunks = (g.bn + kBM - 1) / kBM;
      if (g.splits == 1) {
        for (int c = 0; c < n_chunks; ++c) {
          const int cols = min(kBM, g.bn - c * kBM);
          for (int j = 0; j < cols; j += 16) {
            float v[16];
            tmem_ld16(t_lane + c * kBM + j, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) S[(j + i) * kSLD + row] = v[i];
          }
          named_bar(1, 128);
          apply_epilogue(g, S, c * kBM, cols, m_tile, n_tile, etid);
          named_bar(1, 128);
        }
      } else {
        const size_t tile_id = static_cast<size_t>(m_tile) * g.n_tiles + n_tile;
        const size_t tile_elems = static_cast<size_t>(g.bn) * kBM;
        float* part = g.partial + tile_id * g.splits * tile_elems;
        float* mine = part + split * tile_elems;
        for (int j = 0; j < g.bn; j += 16) {
          float v[16];
          tmem_ld16(t_lane + j, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) __stcg(&mine[(j + i) * kBM + row], v[i]);
        }
        __threadfence();
        named_bar(1, 128);
        if (etid == 0) {
          const int prev = atomicAdd(&g.counters[tile_id], 1);
          hdr->last_flag = (prev == g.splits - 1) ? 1 : 0;
        }
        named_bar(1, 128);
        if (hdr->last_flag) {
          __threadfence();
          for (int c = 0; c < n_chunks; ++c) {
            const int cols = min(kBM, g.bn - c * kBM);
            for (int idx = etid; idx < cols * kBM; idx += 128) {
              const int a = idx & 127, b = idx >> 7;
              const size_t off = static_cast<size_t>(c * kBM + b) * kBM + a;
              float acc = 0.f;
              for (int s = 0; s < g.splits; ++s) acc += __ldcg(&part[s * tile_elems + off]);
              S[b * kSLD + a] = acc;
            }
            named_bar(1, 128);
            apply_epilogue(g, S, c * kBM, cols, m_tile, n_tile, etid);
            named_bar(1, 128);
          }
          if (etid == 0) g.counters[tile_id] = 0;
        }
      }
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

}  // namespace
}  // namespace dfl

namespace dfl {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_operand_map(CUtensorMap* map, const void* base, int elem_bytes, uint64_t k,
                      uint64_t rows, uint64_t zdim, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr || base == nullptr || rows == 0 || zdim == 0 || box_rows == 0 ||
      box_rows > 256)
    return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0) return false;
  cuuint64_t dims[3] = {k, rows, zdim};
  cuuint64_t strides[2] = {k * elem_bytes, k * rows * elem_bytes};
  cuuint32_t box[3] = {128u / static_cast<uint32_t>(elem_bytes), box_rows, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r =
      fn(map, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
         3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

GemmPlan plan_gemm(int m_tiles, int n_rows, int k, int elem_bytes, int num_sms, bool allow_split,
                   int bn_cap) {
  GemmPlan p{};
  const int bk = 128 / elem_bytes;
  const int KT = k / bk;
  const int n16 = (n_rows + 15) / 16 * 16;
  const int cap1 = bn_cap < 256 ? bn_cap : 256;
  if (n16 <= cap1) {
    p.bn = n16; p.n_sub = 1; p.n_tiles = 1;
  } else if (n16 <= bn_cap && n16 <= kMaxBN) {
    p.bn = (n_rows + 31) / 32 * 32; p.n_sub = 2; p.n_tiles = 1;
  } else {
    p.bn = cap1; p.n_sub = 1; p.n_tiles = (n_rows + cap1 - 1) / cap1;
  }
  p.m_tiles = m_tiles;
  const size_t stage = 16384 + static_cast<size_t>(p.bn) * 128;
  const size_t staging = static_cast<size_t>(p.bn < kBM ? p.bn : kBM) * 129 * 4;
  const int ctas_per_sm = p.bn <= 64 ? 2 : 1;
  const size_t budget = (ctas_per_sm == 2 ? 110 * 1024 : 222 * 1024) - 2048;
  int stages = static_cast<int>(budget / stage);
  if (stages > 16) stages = 16;
  if (stages > KT && KT >= 2) stages = KT;
  if (stages < 2) stages = 2;
  while (static_cast<size_t>(stages) * stage < staging) ++stages;
  p.stages = stages;
  p.smem_bytes = 2048 + static_cast<size_t>(stages) * stage;
  int splits = 1;
  if (allow_split) {
    const int tiles = m_tiles * p.n_tiles;
    const int target = num_sms * ctas_per_sm;
    splits = target / (tiles > 0 ? tiles : 1);
    if (splits > KT / 4) splits = KT / 4;
    if (splits > 32) splits = 32;
    if (splits < 1) splits = 1;
  }
  p.kt_per_split = (KT + splits - 1) / splits;
  p.splits = (KT + p.kt_per_split - 1) / p.kt_per_split;
  p.partial_bytes = p.splits > 1 ? static_cast<size_t>(m_tiles) * p.n_tiles * p.splits * p.bn * kBM * 4 : 0;
  return p;
}

cudaError_t launch_gemm(const CUtensorMap& a_map, const CUtensorMap& b_map, const GemmArgs& args,
                        const GemmPlan& plan, cudaStream_t stream, bool pdl) {
  void (*kern)(const CUtensorMap, const CUtensorMap, const GemmArgs, int) =
      args.tf32 ? gemm_tc_kernel<true> : gemm_tc_kernel<false>;
  static bool configured[2][64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  bool& done = configured[args.tf32 ? 1 : 0][dev & 63];
  if (!done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.m_tiles, plan.splits, plan.n_tiles);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, a_map, b_map, args, plan.stages);
}

}  // namespace dfl
