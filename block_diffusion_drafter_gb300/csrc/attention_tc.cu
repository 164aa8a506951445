// Context attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Every block row of every query head attends to all ctx_len[b] + R keys of
// its KV head, with no mask (bidirectional inside the block): the K_i / V_i
// equations of "KV Injection 메커니즘" in "DFlash: Block Diffusion for Flash
// Speculative Decoding 논문 정리", and §3.2 of the marsggbo DFlash page.
//
// One CTA owns the G*R query rows of one (sequence, KV head) and a contiguous
// slice of its keys. Per 128-key tile t:
//   S_t = Q K_t^T  tcgen05.mma, Q and K K-major in shared memory, into one of
//                  two S buffers in TMEM (one query row per TMEM lane = per
//                  softmax thread), so S_{t+1} is computed while the softmax
//                  of tile t runs;
//   softmax        row max / exp2 / row sum are thread-local; the running max
//                  is raised lazily (O in TMEM is rescaled only when the max
//                  grows by more than 2^8), P goes to shared memory as bf16;
//   O += P V_t     tcgen05.mma with V as an MN-major operand, O in TMEM.
// K and V tiles stream in by TMA through two 2-stage rings of their own, so a
// K stage is refilled as soon as its S product is done. Warp 0 issues TMA
// (lane 0 K, lane 1 V), warp 1 the MMAs, warps 2-9 run the softmax (two per
// TMEM lane quarter); a quarter holding no query row only keeps the barrier
// counts. The key slices of one (sequence, KV head) form a thread-block
// cluster whose partial results are merged through distributed shared memory;
// for long contexts with few (sequence, KV head) pairs there are more slices
// than a cluster holds (one per SM), and attn_merge_kernel merges them from
// the workspace.
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"

namespace dfl {
namespace {

constexpr int kTileKeys = 128;
constexpr uint32_t kSub = 128 * 128;     // one 128-row x 128-byte swizzled sub-tile (16 KB)
constexpr int kMaxCluster = 12;  // split-KV CTAs per cluster (the planner never exceeds it)
constexpr float kLog2eTc = 1.4426950408889634f;
constexpr float kLazyRescale = 8.0f;     // log2 units the running max may lag behind

// Softmax warps per TMEM lane quarter: each takes 128 / kParts keys of every
// S tile (and DH / kParts columns of O). Two, not four: with four the
// register budget of 18 warps (96 per thread) spills, and the 32K-context
// attention ran at 0.50 instead of 0.54 of the HBM peak.
constexpr int kParts = 2;
constexpr int kAttnThreads = 64 + 128 * kParts;  // TMA warp, MMA warp, softmax warps

struct AttnSmem {
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t q_full, s_full[2], s_free[2], p_full, o_done;
  uint32_t tmem_base;
  int abort_flag;
  int seq;                  // the sequence this CTA's launch slot takes (longest first)
  float pmax[kParts][128];  // per-part row max of the current tile
  float psum[kParts][128];  // per-part row sums at the end
};


__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
// Byte offset of 16-byte chunk c (of a 128-byte row segment) in row r of a
// 128-byte swizzled sub-tile.
// 2^x by the hardware approximation (ex2.approx, relative error ~2^-22); its
// result is rounded to bf16 for P anyway.
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t swz128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}
__device__ __forceinline__ float2 ld_dsmem_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
// Bounded wait whose outcome is the same on every lane of the warp (the
// warp-collective tcgen05 loads that follow need a converged warp).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity)) != 0;
}

template <int DH>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                   const AttnArgs p) {
  constexpr int NSUB = DH / 64;                      // 64-dim sub-tiles per head
  constexpr uint32_t kQBytes = NSUB * kSub;
  constexpr uint32_t kPBytes = 2 * kSub;             // 128 keys = two 64-key sub-tiles
  constexpr uint32_t kTileBytes = NSUB * kSub;       // K or V of one tile
  constexpr uint32_t kOCol = 256;                    // TMEM columns: S buffers 0 / 128, O 256
  constexpr uint32_t kTmemCols = 512;
  extern __shared__ uint8_t smem_raw[];
  AttnSmem* hdr = reinterpret_cast<AttnSmem*>(smem_raw);
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t base_s = (raw_s + sizeof(AttnSmem) + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_s - raw_s);
  const uint32_t q_s = base_s, p_s = q_s + kQBytes, k_s = p_s + kPBytes, v_s = k_s + 2 * kTileBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sp = blockIdx.x, kvh = blockIdx.y;
  int b = blockIdx.z;   // until the dependency wait: the launch slot (see below)
  int issued = 0;  // producer lanes: tiles whose TMA loads were issued
  const int G = p.n_q_heads / p.n_kv_heads;
  const int n_q = G * p.R;

  // The first tiles of this split's context K/V do not depend on the kernel
  // this one waits for: ask L2 for them now, so that the HBM reads overlap
  // that kernel's tail and this kernel's set-up (a hint only: the TMA loads
  // below read whatever the memory holds after the wait). Rows stay inside
  // this (layer, sequence, KV head) slab of the cache.
  if (threadIdx.x == 64 && p.page_table == nullptr) {
    const int kb0 = sp * p.chunk;
    const size_t slab0 = (static_cast<size_t>(p.layer) * p.max_batch + b) * p.n_kv_heads + kvh;
    for (int t = 0; t < p.prefetch_tiles; ++t) {
      const int r0 = kb0 + t * kTileKeys, r1 = min(r0 + kTileKeys, p.ncap);
      if (r0 >= r1) break;
      const size_t off = (slab0 * p.ncap + r0) * DH;
      const uint32_t bytes = static_cast<uint32_t>(r1 - r0) * DH * 2;
      prefetch_l2_bulk(reinterpret_cast<const __nv_bfloat16*>(p.k_cache) + off, bytes);
      prefetch_l2_bulk(reinterpret_cast<const __nv_bfloat16*>(p.v_cache) + off, bytes);
    }
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&hdr->k_full[i]), 1);
      mbar_init(smem_u32(&hdr->k_empty[i]), 1);
      mbar_init(smem_u32(&hdr->v_full[i]), 1);
      mbar_init(smem_u32(&hdr->v_empty[i]), 1);
      mbar_init(smem_u32(&hdr->s_full[i]), 1);
      mbar_init(smem_u32(&hdr->s_free[i]), kAttnThreads - 64);
    }
    mbar_init(smem_u32(&hdr->q_full), kAttnThreads - 64);
    mbar_init(smem_u32(&hdr->p_full), kAttnThreads - 64);
    mbar_init(smem_u32(&hdr->o_done), 1);
    hdr->abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&hdr->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&k_map);
    tma_prefetch_map(&v_map);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = hdr->tmem_base;
  pdl_launch_dependents();
  pdl_wait();

  // Longest contexts first. The (sequence, KV head) clusters start in the
  // order of their launch slot z = blockIdx.z; in a batch of ragged contexts
  // slot z takes the sequence of rank z by context length (longest first,
  // ties by index), so that the longest clusters start first and the short
  // ones fill in behind them instead of a long one starting last. Equal
  // contexts keep the identity order.
  if (p.B > 1 && p.B <= 64) {
    if (warp == 0) {
      const int l0 = lane < p.B ? p.ctx_len[lane] : -1;
      const int l1 = lane + 32 < p.B ? p.ctx_len[lane + 32] : -1;
      int r0 = 0, r1 = 0;   // ranks of sequences lane and lane + 32
      for (int m = 0; m < p.B; ++m) {
        const int lm = __shfl_sync(0xffffffffu, m < 32 ? l0 : l1, m & 31);
        r0 += (lm > l0 || (lm == l0 && m < lane)) ? 1 : 0;
        r1 += (lm > l1 || (lm == l1 && m < lane + 32)) ? 1 : 0;
      }
      if (lane < p.B && r0 == b) hdr->seq = lane;
      if (lane + 32 < p.B && r1 == b) hdr->seq = lane + 32;
    }
    __syncthreads();
    b = hdr->seq;
  }

  // the block's keys: rows 0..gamma_b[b] (clamped to the block), else all R
  const int r_b = p.gamma_b == nullptr ? p.R : min(max(p.gamma_b[b], 1), p.R - 1) + 1;
  const int n_keys = p.ctx_len[b] + r_b;
  // This sequence's keys are split evenly over the splits (whole 128-key
  // tiles; p.chunk is the split of the longest context). In a ragged batch a
  // short context then has short splits, instead of its first splits taking
  // all of it while the rest idle in the cluster until its merge.
  const int chunk_b = ((n_keys + p.splits - 1) / p.splits + kTileKeys - 1) / kTileKeys * kTileKeys;
  const int k_begin = sp * chunk_b;
  const int k_end = (sp == p.splits - 1) ? n_keys : min(n_keys, (sp + 1) * chunk_b);
  const int nt = k_end > k_begin ? (k_end - k_begin + kTileKeys - 1) / kTileKeys : 0;
  const int slab = (p.layer * p.max_batch + b) * p.n_kv_heads + kvh;
  volatile int* abort_flag = &hdr->abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producers
    // lane 0 streams K tiles, lane 1 V tiles, each through its own ring
    if (lane < 2) {
      const bool is_v = lane == 1;
      const CUtensorMap* map = is_v ? &v_map : &k_map;
      const uint32_t ring = is_v ? v_s : k_s;
      const uint64_t pol = l2_evict_first();
      // box coordinates of tile t: (y, z) of the contiguous cache slab or of its page
      auto coords = [&](int t, int& y, int& z) -> bool {
        const int kb = k_begin + t * kTileKeys;
        z = slab;
        y = kb;
        if (p.page_table != nullptr) {
          const int pg = p.page_table[static_cast<size_t>(b) * p.pages_per_seq + kb / kPageKeys];
          if (pg < 0 || pg >= p.n_pages) return false;
          z = (p.layer * p.n_pages + pg) * p.n_kv_heads + kvh;
          y = 0;
        }
        return true;
      };
      for (int t = 0; t < nt; ++t) {
        const int st = t & 1, u = t >> 1;
        const uint32_t empty = smem_u32(is_v ? &hdr->v_empty[st] : &hdr->k_empty[st]);
        if (u > 0 && !mbar_wait(empty, (u - 1) & 1)) {
          report(p.dev_status, DFLASH_ERR_TIMEOUT);
          atomicExch(&hdr->abort_flag, 1);
          break;
        }
        if (*abort_flag) break;
        const uint32_t bar = smem_u32(is_v ? &hdr->v_full[st] : &hdr->k_full[st]);
        const uint32_t dst = ring + st * kTileBytes;
        int y, z;
        if (!coords(t, y, z)) {  // the tile is a page outside the pool
          report(p.dev_status, DFLASH_ERR_CAPACITY);
          z = p.layer * p.n_pages * p.n_kv_heads + kvh;   // page 0
          y = 0;
        }
        mbar_expect_tx(bar, kTileBytes);
#pragma unroll
        for (int j = 0; j < NSUB; ++j) tma_load_3d(dst + j * kSub, map, bar, 64 * j, y, z, pol);
        issued = t + 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // order: S_0, then per tile t: S_{t+1} (as soon as K_{t+1} is in and its
    // S buffer was read), P_t V_t (once the softmax wrote P_t)
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc(128, kTileKeys, kFmtBF16);
      const uint32_t idesc_o = make_idesc(128, DH, kFmtBF16, 1);
      auto issue_s = [&](int t) -> bool {
        const int st = t & 1, u = t >> 1;
        if (!mbar_wait(smem_u32(&hdr->k_full[st]), u & 1)) return false;
        if (t >= 2 && !mbar_wait(smem_u32(&hdr->s_free[st]), (u - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t kt = k_s + st * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < DH / 16; ++ks) {
          const uint32_t off = (ks >> 2) * kSub + (ks & 3) * 32;
          tc_mma_f16(tmem + st * kTileKeys, sw128_desc(q_s + off), sw128_desc(kt + off), idesc_s,
                     ks > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(&hdr->s_full[st]));
        tc_commit(smem_u32(&hdr->k_empty[st]));
        return true;
      };
      bool ok = nt == 0 || (mbar_wait(smem_u32(&hdr->q_full), 0) && issue_s(0));
      for (int t = 0; ok && t < nt; ++t) {
        if (t + 1 < nt && !issue_s(t + 1)) { ok = false; break; }
        const int st = t & 1, u = t >> 1;
        ok = mbar_wait(smem_u32(&hdr->p_full), t & 1) && mbar_wait(smem_u32(&hdr->v_full[st]), u & 1);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vt = v_s + st * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < kTileKeys / 16; ++ks) {
          const uint64_t a = sw128_desc(p_s + (ks >> 2) * kSub + (ks & 3) * 32);
          const uint64_t bd = sw128_desc_mn(vt + ks * 2048, kSub, 1024);
          tc_mma_f16(tmem + kOCol, a, bd, idesc_o, (t > 0 || ks > 0) ? 1u : 0u);
        }
        tc_commit(smem_u32(&hdr->o_done));
        tc_commit(smem_u32(&hdr->v_empty[st]));
      }
      if (!ok) {
        report(p.dev_status, DFLASH_ERR_TIMEOUT);
        atomicExch(&hdr->abort_flag, 1);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    // Softmax warps: TMEM lane quarter (warp % 4) gives the query row; `part`
    // picks keys HK*part..+HK-1 of each S tile and columns HO*part..+HO-1 of
    // O. A quarter without query rows (all q >= n_q) computes nothing.
    const int q = (warp & 3) * 32 + lane;
    const int part = (warp - 2) >> 2;
    const bool live = (warp & 3) * 32 < n_q;   // warp-uniform
    const uint32_t t_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const size_t hq_stride = static_cast<size_t>(p.n_q_heads) * DH;
    const int gq = q / p.R, iq = q % p.R;
    const __nv_bfloat16* qg = reinterpret_cast<const __nv_bfloat16*>(p.q);
    const size_t row_off = (static_cast<size_t>(b) * p.R + iq) * hq_stride + static_cast<size_t>(kvh * G + gq) * DH;
    constexpr int QC = DH / 8;          // 16-byte chunks of one Q row
    // this thread's part of Q row q into the swizzled K-major tile (rows >= n_q zero)
#pragma unroll
    for (int c = part * (QC / kParts); c < (part + 1) * (QC / kParts); ++c) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (q < n_q) v = *reinterpret_cast<const uint4*>(qg + row_off + c * 8);
      st_shared_v4(q_s + (c >> 3) * kSub + swz128(q, c & 7), v);
    }
    fence_proxy_async();
    mbar_arrive(smem_u32(&hdr->q_full));

    const float scale = rsqrtf(static_cast<float>(DH)) * kLog2eTc;
    constexpr int HK = kTileKeys / kParts;   // keys per part
    constexpr int HO = DH / kParts;          // O columns per part
    constexpr int kBarThreads = 32 * kParts; // the warps of one lane quarter
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int t = 0; t < nt; ++t) {
      const int j = t & 1;
      const int kb = k_begin + t * kTileKeys;
      const int nvalid = min(kTileKeys, k_end - kb);
      const int nv_part = min(HK, max(0, nvalid - part * HK));
      if (!warp_wait(smem_u32(&hdr->s_full[j]), (t >> 1) & 1)) { ok = false; break; }
      float sv[HK];
      if (live) {
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < HK; c0 += 16) tmem_ld16(t_row + j * kTileKeys + part * HK + c0, sv + c0);
        tmem_ld_wait();
      }
      // S_t is in registers: its buffer may take S_{t+2}
      tc_fence_before();
      mbar_arrive(smem_u32(&hdr->s_free[j]));
      float m_use = m_run;
      bool rescale = false;
      float m_new = m_run;
      if (live) {
        if (nv_part < HK) {
#pragma unroll
          for (int i = 0; i < HK; ++i)
            if (i >= nv_part) sv[i] = -INFINITY;
        }
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = sv[i];
#pragma unroll
        for (int i = 8; i < HK; ++i) m8[i & 7] = fmaxf(m8[i & 7], sv[i]);
        float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                         fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        // all parts of the row agree on its max
        hdr->pmax[part][q] = mx;
        named_bar(2 + (warp & 3), kBarThreads);
        mx = hdr->pmax[0][q];
#pragma unroll
        for (int k = 1; k < kParts; ++k) mx = fmaxf(mx, hdr->pmax[k][q]);
        mx *= scale;
        m_new = fmaxf(m_run, mx);
        rescale = (m_run == -INFINITY) || (m_new > m_run + kLazyRescale);
        m_use = rescale ? m_new : m_run;
      }
      // the previous P . V must be done before P is rewritten or O rescaled;
      // every softmax warp waits for it, so that no warp runs ahead and
      // arrives on p_full for a later tile while this one is still open
      if (t > 0) {
        if (!warp_wait(smem_u32(&hdr->o_done), (t - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (live && __any_sync(0xffffffffu, rescale)) {
          const float alpha = rescale ? exp2_approx(m_run - m_new) : 1.f;
          if (rescale) l_run *= alpha;
          float ov[HO];
#pragma unroll
          for (int c0 = 0; c0 < HO; c0 += 16) tmem_ld16(t_row + kOCol + part * HO + c0, ov + c0);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < HO; ++i) ov[i] *= alpha;
#pragma unroll
          for (int c0 = 0; c0 < HO; c0 += 16) tmem_st16(t_row + kOCol + part * HO + c0, ov + c0);
          tmem_st_wait();
        }
      }
      m_run = m_use;
      if (nvalid < kTileKeys) {
        // keys past the end of the slice: zero their V rows (cache rows beyond
        // the context may hold anything, and 0 * NaN would poison O)
        if (!warp_wait(smem_u32(&hdr->v_full[j]), (t >> 1) & 1)) { ok = false; break; }
        if (q >= nvalid) {
          const uint32_t vt = v_s + j * kTileBytes;
#pragma unroll
          for (int jj = 0; jj < NSUB; ++jj)
#pragma unroll
            for (int c = part * (8 / kParts); c < (part + 1) * (8 / kParts); ++c)
              st_shared_v4(vt + jj * kSub + q * 128 + c * 16, make_uint4(0u, 0u, 0u, 0u));
        }
      }
      if (live) {
        // P = 2^(s * scale - m) as bf16 into the K-major P tile (keys HK*part..)
        float ls[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) ls[i] = 0.f;
#pragma unroll
        for (int c = 0; c < HK / 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            const float p0 = exp2_approx(fmaf(sv[c * 8 + i], scale, -m_use));
            const float p1 = exp2_approx(fmaf(sv[c * 8 + i + 1], scale, -m_use));
            ls[i] += p0;
            ls[i + 1] += p1;
            w[i >> 1] = pack2_bf16(p0, p1);
          }
          const int key = part * HK + c * 8;
          st_shared_v4(p_s + (key >> 6) * kSub + swz128(q, (key & 63) >> 3), make_uint4(w[0], w[1], w[2], w[3]));
        }
        l_run += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      }
      fence_proxy_async();
      tc_fence_before();
      mbar_arrive(smem_u32(&hdr->p_full));
    }
    if (ok && nt > 0) {
      ok = warp_wait(smem_u32(&hdr->o_done), (nt - 1) & 1);
      tc_fence_after();
    }
    if (!ok) {
      report(p.dev_status, DFLASH_ERR_TIMEOUT);
      atomicExch(&hdr->abort_flag, 1);
    }
    // row sum over the parts (same running max), in a fixed order
    hdr->psum[part][q] = l_run;
    named_bar(2 + (warp & 3), kBarThreads);
    float l_row = hdr->psum[0][q];
#pragma unroll
    for (int k = 1; k < kParts; ++k) l_row += hdr->psum[k][q];
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    const bool have = ok && nt > 0 && live;
    float ov[HO];
    if (have) {  // warp-uniform
#pragma unroll
      for (int c0 = 0; c0 < HO; c0 += 16) tmem_ld16(t_row + kOCol + part * HO + c0, ov + c0);
      tmem_ld_wait();
    }
    if (p.splits == 1) {
      if (have && q < n_q) {
        const float inv = l_row > 0.f ? 1.f / l_row : 0.f;
#pragma unroll
        for (int c0 = 0; c0 < HO; c0 += 8) {
          float x[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = ov[c0 + i] * inv;
          uint4 w;
          w.x = pack2_bf16(x[0], x[1]); w.y = pack2_bf16(x[2], x[3]);
          w.z = pack2_bf16(x[4], x[5]); w.w = pack2_bf16(x[6], x[7]);
          *reinterpret_cast<uint4*>(out + row_off + part * HO + c0) = w;
          if (p.out_lo_off) {
            const __nv_bfloat162* hw = reinterpret_cast<const __nv_bfloat162*>(&w);
            uint4 lw;
            uint32_t* l = reinterpret_cast<uint32_t*>(&lw);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 hf = __bfloat1622float2(hw[i]);
              l[i] = pack2_bf16(x[2 * i] - hf.x, x[2 * i + 1] - hf.y);
            }
            *reinterpret_cast<uint4*>(out + p.out_lo_off + row_off + part * HO + c0) = lw;
          }
        }
      }
    } else if (p.merge_global) {
      // this split's unnormalised O row and (m, l) to its workspace slot
      if (q < n_q) {
        float* slot = p.partials + (static_cast<size_t>(b * p.n_kv_heads + kvh) * p.splits + sp) *
                                       attn_slot_floats(DH);
        float4* orow = reinterpret_cast<float4*>(slot + static_cast<size_t>(q) * DH + part * HO);
#pragma unroll
        for (int i = 0; i < HO; i += 4)
          orow[i / 4] = have ? make_float4(ov[i], ov[i + 1], ov[i + 2], ov[i + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (part == 0)
          reinterpret_cast<float2*>(slot + static_cast<size_t>(128) * DH)[q] =
              have ? make_float2(m_run, l_row) : make_float2(-INFINITY, 0.f);
      }
    } else {
      // park the unnormalised O row and (m, l) for the cluster merge
      float* po = reinterpret_cast<float*>(base + (k_s - base_s));
      constexpr int PLD = DH + 4;
#pragma unroll
      for (int i = 0; i < HO; i += 4)
        *reinterpret_cast<float4*>(&po[q * PLD + part * HO + i]) =
            have ? make_float4(ov[i], ov[i + 1], ov[i + 2], ov[i + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (part == 0) {
        float2* ml = reinterpret_cast<float2*>(po + 128 * PLD);
        ml[q] = have ? make_float2(m_run, l_row) : make_float2(-INFINITY, 0.f);
      }
    }
    tc_fence_before();
  }

  if (p.splits > 1 && !p.merge_global) {
    // Split-KV merge inside the cluster: CTA r merges a slice of the query
    // rows, reading every split's O row and (m, l) through distributed shared
    // memory in ascending split order, each weighted by 2^(m_s - M) / L. A
    // thread requests all of its remote values at once (one round trip), and
    // arrives on the closing cluster barrier as soon as its reads are done.
    cluster_sync();
    constexpr int PLD = DH + 4;
    const uint32_t po_u = k_s, ml_u = k_s + 128 * PLD * 4;
    const int S = p.splits;
    const int rank = static_cast<int>(cluster_ctarank());
    const int per = (n_q + S - 1) / S;
    const int r0 = rank * per, r1 = min(n_q, r0 + per);
    const int nrows = r1 > r0 ? r1 - r0 : 0;
    constexpr int D4 = DH / 4;
    const size_t hq_stride = static_cast<size_t>(p.n_q_heads) * DH;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
    for (int it = threadIdx.x; it < nrows * D4; it += blockDim.x) {
      const int r = it / D4, qr = r0 + r, d = (it % D4) * 4;
      const uint32_t off = po_u + static_cast<uint32_t>((qr * PLD + d) * 4);
      float4 v[kMaxCluster];
      float2 ml[kMaxCluster];
#pragma unroll
      for (int s2 = 0; s2 < kMaxCluster; ++s2) {
        if (s2 < S) {
          ml[s2] = ld_dsmem_f2(mapa_shared(ml_u + qr * 8, s2));
          v[s2] = ld_dsmem_f4(mapa_shared(off, s2));
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int s2 = 0; s2 < kMaxCluster; ++s2)
        if (s2 < S && ml[s2].y > 0.f) M = fmaxf(M, ml[s2].x);
      float L = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < kMaxCluster; ++s2)
        if (s2 < S) L += ml[s2].y * (ml[s2].y > 0.f ? exp2f(ml[s2].x - M) : 0.f);
      const float inv = L > 0.f ? 1.f / L : 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s2 = 0; s2 < kMaxCluster; ++s2) {
        if (s2 < S) {
          const float w = (ml[s2].y > 0.f ? exp2f(ml[s2].x - M) : 0.f) * inv;
          acc.x += v[s2].x * w; acc.y += v[s2].y * w; acc.z += v[s2].z * w; acc.w += v[s2].w * w;
        }
      }
      const int g = qr / p.R, i = qr % p.R;
      const size_t oi = (static_cast<size_t>(b) * p.R + i) * hq_stride + static_cast<size_t>(kvh * G + g) * DH + d;
      store_hilo(out, oi, p.out_lo_off, acc.x);
      store_hilo(out, oi + 1, p.out_lo_off, acc.y);
      store_hilo(out, oi + 2, p.out_lo_off, acc.z);
      store_hilo(out, oi + 3, p.out_lo_off, acc.w);
    }
    cluster_arrive();
  }
  __syncthreads();
  // after a timeout, no TMA load of this CTA may still be landing when it
  // exits: each producer lane waits (bounded) for the last two tiles of its
  // ring; earlier tiles of a stage completed before the stage was refilled
  if (warp == 0 && lane < 2 && *abort_flag) {
    for (int t = issued > 2 ? issued - 2 : 0; t < issued; ++t)
      mbar_wait(smem_u32(lane == 1 ? &hdr->v_full[t & 1] : &hdr->k_full[t & 1]), (t >> 1) & 1);
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // the peers may still be reading this CTA's partial rows
  if (p.splits > 1 && !p.merge_global) cluster_wait();
}

// Merge of the split partials written to the workspace: CTA (x, kvh, b)
// takes query rows 4x..4x+3 of one (sequence, KV head), a warp per row, each
// lane DH/32 of its columns. Lane s holds split s's (m, l) (s, s+32, ... for
// more splits); the running max M is a warp reduction, the weights
// 2^(m_s - M) / L and the column sums are taken in ascending split order, the
// same arithmetic as the cluster merge. The O rows of the first kMergeBatch
// splits are requested together with the (m, l) pairs, so a row costs one L2
// round trip for up to kMergeBatch splits.
constexpr int kMergeBatch = 24;
template <int DH>
__global__ void __launch_bounds__(128) attn_merge_kernel(const AttnArgs p) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int DPT = DH / 32;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int G = p.n_q_heads / p.n_kv_heads;
  const int n_q = G * p.R;
  const int qr = blockIdx.x * 4 + static_cast<int>(threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (qr >= n_q) return;   // warp-uniform: whole warps leave
  const int S = p.splits;
  const size_t slot_f = attn_slot_floats(DH);
  const float* base = p.partials + static_cast<size_t>(b * p.n_kv_heads + kvh) * S * slot_f;
  const float2* ml = reinterpret_cast<const float2*>(base + static_cast<size_t>(128) * DH) + qr;
  const float* row = base + static_cast<size_t>(qr) * DH + lane * DPT;
  auto load_o = [&](int s2, float* x) {
    if (DPT == 4) {
      const float4 t = __ldcg(reinterpret_cast<const float4*>(row + s2 * slot_f));
      x[0] = t.x; x[1 % DPT] = t.y; x[2 % DPT] = t.z; x[3 % DPT] = t.w;
    } else {
      const float2 t = __ldcg(reinterpret_cast<const float2*>(row + s2 * slot_f));
      x[0] = t.x; x[1 % DPT] = t.y;
    }
  };
  float x[kMergeBatch][DPT];
#pragma unroll
  for (int u = 0; u < kMergeBatch; ++u)
    if (u < S) load_o(u, x[u]);
  // (m, l) of splits lane, lane + 32, ... (at most kAttnMaxSlots splits)
  constexpr int kPer = (kAttnMaxSlots + 31) / 32;
  float2 mv[kPer];
  float M = -INFINITY;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int s2 = lane + 32 * k;
    mv[k] = s2 < S ? __ldcg(ml + s2 * (slot_f / 2)) : make_float2(-INFINITY, 0.f);
    if (mv[k].y > 0.f) M = fmaxf(M, mv[k].x);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float wk[kPer];   // 2^(m_s - M) of this lane's splits
#pragma unroll
  for (int k = 0; k < kPer; ++k) wk[k] = mv[k].y > 0.f ? exp2f(mv[k].x - M) : 0.f;
  // split s2's weight and l, broadcast from the lane that holds it (one
  // shuffle while the splits fit in a warp's lanes)
  auto from_lane = [&](const float* v, int s2) {
    float r = __shfl_sync(0xffffffffu, v[0], s2 & 31);
    if (S > 32) {   // warp-uniform
#pragma unroll
      for (int k = 1; k < kPer; ++k) {
        const float t = __shfl_sync(0xffffffffu, v[k], s2 & 31);
        if ((s2 >> 5) == k) r = t;
      }
    }
    return r;
  };
  float lk[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) lk[k] = mv[k].y;
  float L = 0.f;
  for (int s2 = 0; s2 < S; ++s2) L = fmaf(from_lane(lk, s2), from_lane(wk, s2), L);   // ascending order
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float acc[DPT];
#pragma unroll
  for (int i = 0; i < DPT; ++i) acc[i] = 0.f;
  for (int s0 = 0; s0 < S; s0 += kMergeBatch) {
    if (s0 > 0) {
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u)
        if (s0 + u < S) load_o(s0 + u, x[u]);
    }
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const float w = from_lane(wk, s0 + u) * inv;
      if (s0 + u < S) {
#pragma unroll
        for (int i = 0; i < DPT; ++i) acc[i] += x[u][i] * w;
      }
    }
  }
  const int g = qr / p.R, i = qr % p.R;
  const size_t hq_stride = static_cast<size_t>(p.n_q_heads) * DH;
  const size_t oi = (static_cast<size_t>(b) * p.R + i) * hq_stride + static_cast<size_t>(kvh * G + g) * DH + lane * DPT;
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
  for (int k = 0; k < DPT; ++k) store_hilo(out, oi + k, p.out_lo_off, acc[k]);
}

}  // namespace
}  // namespace dfl

namespace dfl {

cudaError_t launch_attention_tc(const AttnArgs& a_in, cudaStream_t stream, bool pdl) {
  AttnArgs a = a_in;
  // K/V tiles per split asked of L2 before the dependency wait: off by
  // default. Measured at 32768 keys: attention calls back to back in a graph
  // 28.3 -> 27.3 us with 3 tiles, but inside the drafting step, where the
  // QKV projection before it streams weights at the HBM peak, no gain (C3
  // step 835 vs 840 us). DFLASH_ATTN_PREFETCH sets the count (tuning).
  static int prefetch = -1;
  if (prefetch < 0) {
    const char* e = getenv("DFLASH_ATTN_PREFETCH");
    prefetch = e != nullptr ? atoi(e) : 0;
    if (prefetch < 0) prefetch = 0;
  }
  a.prefetch_tiles = prefetch;
  if (a.head_dim != 64 && a.head_dim != 128) return cudaErrorInvalidValue;
  if ((a.n_q_heads / a.n_kv_heads) * a.R > 128) return cudaErrorInvalidValue;
  const bool global = a.splits > 1 && a.merge_global;
  if (!global && a.splits > kMaxCluster) return cudaErrorInvalidValue;
  if (global && (a.partials == nullptr || a.B * a.n_kv_heads * a.splits > kAttnMaxSlots))
    return cudaErrorInvalidValue;
  // one tensor map per cache over all layers: [L * max_batch * Hkv][Ncap][Dh],
  // or for page pools [L * n_pages * Hkv][kPageKeys][Dh] (a tile is a page)
  CUtensorMap km, vm;
  const bool paged = a.page_table != nullptr;
  const uint64_t slabs = static_cast<uint64_t>(a.n_layers) * (paged ? a.n_pages : a.max_batch) * a.n_kv_heads;
  const uint64_t rows = paged ? kPageKeys : a.ncap;
  if (!make_operand_map(&km, a.k_cache, 2, a.head_dim, rows, slabs, kTileKeys) ||
      !make_operand_map(&vm, a.v_cache, 2, a.head_dim, rows, slabs, kTileKeys))
    return cudaErrorInvalidValue;
  const int nsub = a.head_dim / 64;
  const size_t smem = sizeof(AttnSmem) + 1024 + static_cast<size_t>(nsub) * kSub + 2 * kSub +
                      2 * static_cast<size_t>(2 * nsub) * kSub + 4096;  // + slack past the ring
  void (*kern)(const CUtensorMap, const CUtensorMap, const AttnArgs) =
      a.head_dim == 128 ? attn_tc_kernel<128> : attn_tc_kernel<64>;
  static bool configured[2][64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  bool& done = configured[a.head_dim == 128][dev & 63];
  if (!done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.splits, a.n_kv_heads, a.B);
  cfg.blockDim = dim3(kAttnThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (a.splits > 1 && !global) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = a.splits;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, km, vm, a);
}

cudaError_t launch_attention_merge(const AttnArgs& a, cudaStream_t stream, bool pdl) {
  if (!(a.bf16 && a.splits > 1 && a.merge_global)) return cudaSuccess;
  if (a.head_dim != 64 && a.head_dim != 128) return cudaErrorInvalidValue;
  // merge of the workspace partials: 4 query rows per CTA
  cudaLaunchConfig_t mc = {};
  const int n_q = (a.n_q_heads / a.n_kv_heads) * a.R;
  mc.gridDim = dim3((n_q + 3) / 4, a.n_kv_heads, a.B);
  mc.blockDim = dim3(128, 1, 1);
  mc.stream = stream;
  cudaLaunchAttribute mattr[1];
  mattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  mattr[0].val.programmaticStreamSerializationAllowed = 1;
  mc.attrs = pdl ? mattr : nullptr;
  mc.numAttrs = pdl ? 1 : 0;
  return a.head_dim == 128 ? cudaLaunchKernelEx(&mc, attn_merge_kernel<128>, a)
                           : cudaLaunchKernelEx(&mc, attn_merge_kernel<64>, a);
}

}  // namespace dfl
