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
// Split-K runs as a thread-block cluster per output tile: the partial tiles
// meet in distributed shared memory and are summed in a fixed split order
// (deterministic; no float atomics, no global partial buffers).
#include <stdio.h>
#include <stdlib.h>

#include "common.cuh"
#include "internal.h"

#include <cudaTypedefs.h>

namespace dfl {

namespace {

constexpr int kSLD = 129;  // staging row stride (floats): conflict-free both ways
constexpr int kMaxSplitK = 8;  // split-K CTAs per cluster (portable cluster size)
// barriers + token table, plus slack to align the tile ring to 1024 bytes
constexpr size_t kSmemHeaderBytes = 4608;

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ void store_out(void* out, int bf16, size_t idx, float v) {
  if (bf16)
    reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(out)[idx] = v;
}

// Applies the epilogue to one staged chunk: S[b * kSLD + a] holds C for
// A-row a (0..127) and B-row col0 + b (0 <= b < cols) of tile (m_tile, n_tile).
// Runs on the 128 epilogue threads (etid 0..127). Every op works in batches
// of a few elements per thread: all global loads of a batch are issued
// before any of its stores, so the loads overlap instead of serialising
// behind possibly-aliasing stores. The generic loop takes batches of
// epi_batch() elements: 2 for narrow tiles (a few tokens; larger batches cost
// registers and code, and a drafting step at batch 1 ran slower with them:
// 758 vs 754 us with 4, 799 us with 8), 4 for the wide instances. The wide
// decode instances of the residual add and of QKV/KV, where every thread
// owns one feature across many tokens, have loops of their own.
template <int kOp, bool kWide>
__host__ __device__ constexpr int epi_batch() {
  return kWide && (kOp == EPI_QKV || kOp == EPI_KV || kOp == EPI_ADD_F32) ? 4 : 2;
}
// Whether an epilogue op has a separate wide-tile instance.
constexpr bool has_wide(int op) { return op == EPI_QKV || op == EPI_KV || op == EPI_ADD_F32; }

struct TokInfo {
  int pos[kBM];       // cache position of the chunk's token x, -1 = skip
  int seq[kBM];       // sequence of token x
  float rstd[kMaxBN]; // folded RMSNorm scale of the tile's token x (1 when not folded)
};

__device__ __forceinline__ float gain_at(const void* g, int bf16, int i) {
  return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(g)[i])
              : reinterpret_cast<const float*>(g)[i];
}

// Folded RMSNorm scale 1 / sqrt(mean(h^2) + eps) of tokens tok0 .. tok0+n-1
// into out[0 .. n), from their per-128-feature partial sums of squares: one
// thread per token sums its slots in ascending order, eight 16-byte loads in
// flight at a time (the sums are latency-bound, not bandwidth-bound). Tokens
// past n_tok get 1. Runs on the 128 epilogue threads.
__device__ __forceinline__ void folded_rstd(const Epi& e, float* out, int tok0, int n, int etid) {
  for (int t = etid; t < n; t += 128) {
    const int tok = tok0 + t;
    float r = 1.f;
    if (tok < e.n_tok) {
      const float* src = e.ss_in + static_cast<size_t>(tok) * e.n_ss;
      float ss = 0.f;
      int k = 0;
      if ((e.n_ss & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
        const float4* s4 = reinterpret_cast<const float4*>(src);
        const int n4 = e.n_ss >> 2;
        for (int k4 = 0; k4 < n4; k4 += 8) {
          float4 v[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = k4 + i < n4 ? s4[k4 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int i = 0; i < 8; ++i) ss += ((v[i].x + v[i].y) + v[i].z) + v[i].w;
        }
        k = e.n_ss;
      }
      for (; k < e.n_ss; ++k) ss += src[k];
      r = 1.0f / sqrtf(ss / static_cast<float>(e.d_model) + e.eps);
    }
    out[t] = r;
  }
}

// Whether the kernel computes the folded-norm scales of the whole tile (one
// per B row) while the main loop runs, instead of per chunk in the epilogue.
__device__ __forceinline__ bool rstd_per_tile(const GemmArgs& g) {
  return g.epi.ss_in != nullptr && g.swap != 0 && g.bn <= kMaxBN;
}

template <int kOp, bool kWide>
__device__ void apply_epilogue(const GemmArgs& g, const float* S, TokInfo* ti, int col0, int cols,
                               int m_tile, int n_tile, int etid) {
  const Epi& e = g.epi;
  const int total = cols * kBM;
  const bool tok_cols = g.swap != 0;  // tokens along B rows (columns of S)
  // rstd[x]: folded-norm scale of the chunk's token x
  const bool pre = rstd_per_tile(g);
  const float* rstd = ti->rstd + (pre ? col0 : 0);
  if (e.ss_in != nullptr && !pre)
    folded_rstd(e, ti->rstd, tok_cols ? n_tile * g.bn + col0 : m_tile * kBM, tok_cols ? cols : kBM, etid);
  if (kOp == EPI_QKV || kOp == EPI_KV || (e.ss_in != nullptr && !pre)) {
    const int nloc = tok_cols ? cols : kBM;
    for (int x = etid; x < nloc; x += 128) {
      const int tok = tok_cols ? n_tile * g.bn + col0 + x : m_tile * kBM + x;
      int pos = -1, seq = 0;
      if ((kOp == EPI_QKV || kOp == EPI_KV) && tok < e.n_tok) {
        seq = tok / e.rows_per_seq;
        const int t = tok - seq * e.rows_per_seq;
        const int base = e.ctx_len[seq];
        if (kOp == EPI_QKV) {
          pos = base + t;
          if (pos >= e.ncap) { report(g.dev_status, DFLASH_ERR_CAPACITY); pos = -1; }
        } else {
          const int nn = e.n_new[seq];
          if (t < nn && base + nn <= e.ncap - e.reserve) pos = base + t;
        }
        // paged caches: the slot of the token table holds the row's page
        if (pos >= 0 && e.page_table != nullptr) {
          const int pg = e.page_table[static_cast<size_t>(seq) * e.pages_per_seq + pos / kPageKeys];
          if (pg < 0 || pg >= e.n_pages) {
            report(g.dev_status, DFLASH_ERR_CAPACITY);
            pos = -1;
          } else {
            seq = pg;
          }
        }
      }
      ti->pos[x] = pos;
      ti->seq[x] = seq;
    }
    named_bar(1, 128);
  }
  switch (kOp) {
    case EPI_STORE:
    case EPI_ADD_F32:
    case EPI_FUSE: {
      // producer of a folded norm (swap orientation): this thread's feature is
      // m_tile * 128 + etid for every element it touches
      const float gx = kOp == EPI_ADD_F32 && e.xg_out != nullptr && m_tile * kBM + etid < e.n_feat
                           ? gain_at(e.xg_gain, e.xg_bf16, m_tile * kBM + etid)
                           : 0.f;
      constexpr int kB = epi_batch<kOp, kWide>();
      if constexpr (kOp == EPI_ADD_F32 && kWide) {
        // (wide residual-add tiles are decode tiles: weights along A rows)
        // This thread's feature is fixed (a = etid). Pass 1 adds the residual
        // to the staged accumulator in place, with 24 tokens' loads in flight
        // at a time; pass 2 stores h_new (and g (.) h_new) token by token
        // from shared memory: a short loop instead of an unrolled batch, whose
        // code would not stay in the instruction cache.
        const int a = etid, feat = m_tile * kBM + a;
        float* h = reinterpret_cast<float*>(e.out);
        float* Sw = const_cast<float*>(S);
        const int tok0 = n_tile * g.bn + col0;
        const int nb = min(cols, e.n_tok - tok0);   // valid tokens of the chunk
        if (e.xg_out != nullptr) {
          // output row of g (.) h_new per token (-1: none), once per chunk
          for (int x = etid; x < cols; x += 128) {
            const int tok = tok0 + x;
            int row = tok < e.n_tok ? tok : -1;
            if (row >= 0 && e.xg_mask_rows) {
              const int i = tok % e.rows_per_seq;
              row = i == 0 ? -1 : (tok / e.rows_per_seq) * e.gamma + i - 1;
            }
            ti->pos[x] = row;
          }
          named_bar(1, 128);
        }
        if (feat < e.n_feat) {
          constexpr int NB = 24;
          for (int b0 = 0; b0 < nb; b0 += NB) {
            float r[NB];
#pragma unroll
            for (int u = 0; u < NB; ++u)
              r[u] = b0 + u < nb ? h[static_cast<size_t>(tok0 + b0 + u) * e.ld + feat] : 0.f;
#pragma unroll
            for (int u = 0; u < NB; ++u) {
              const int b = b0 + u;
              if (b < nb) {
                float v = Sw[b * kSLD + a];
                if (e.ss_in != nullptr) v *= rstd[b];
                Sw[b * kSLD + a] = r[u] + v;
              }
            }
          }
#pragma unroll 2
          for (int b = 0; b < nb; ++b) {
            const float hn = Sw[b * kSLD + a];
            h[static_cast<size_t>(tok0 + b) * e.ld + feat] = hn;
            if (e.xg_out != nullptr) {
              const int row = ti->pos[b];
              if (row >= 0) {
                const size_t xi = static_cast<size_t>(row) * e.d_model + feat;
                const float xv = gx * hn;
                if (e.xg_bf16)
                  store_hilo(reinterpret_cast<__nv_bfloat16*>(e.xg_out), xi, e.lo_off, xv);
                else
                  reinterpret_cast<float*>(e.xg_out)[xi] = xv;
              }
              Sw[b * kSLD + a] = hn * hn;
            }
          }
        }
      }
      if constexpr (!(kOp == EPI_ADD_F32 && kWide))
      for (int base = etid; base < total; base += 128 * kB) {
        float v[kB], r[kB];
        size_t o[kB];
        bool ok[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          const int idx = base + u * 128;
          int a, b;
          if (g.swap) { a = idx & 127; b = idx >> 7; } else { b = idx % cols; a = idx / cols; }
          const int feat = g.swap ? m_tile * kBM + a : n_tile * g.bn + col0 + b;
          const int tok = g.swap ? n_tile * g.bn + col0 + b : m_tile * kBM + a;
          ok[u] = idx < total && tok < e.n_tok && feat < e.n_feat;
          v[u] = ok[u] ? S[b * kSLD + a] : 0.f;
          if (e.ss_in != nullptr && ok[u]) v[u] *= rstd[tok_cols ? b : a];
          o[u] = static_cast<size_t>(tok) * e.ld + feat;
        }
        if (kOp == EPI_ADD_F32) {
#pragma unroll
          for (int u = 0; u < kB; ++u)
            r[u] = ok[u] ? reinterpret_cast<const float*>(e.out)[o[u]] : 0.f;
#pragma unroll
          for (int u = 0; u < kB; ++u) {
            if (!ok[u]) continue;
            const float hn = r[u] + v[u];
            reinterpret_cast<float*>(e.out)[o[u]] = hn;
            if (e.xg_out != nullptr) {
              // folded RMSNorm of the next projection: g (.) h_new and h_new^2
              const int idx = base + u * 128;
              const int a = idx & 127, b = idx >> 7;   // swap orientation
              const int tok = n_tile * g.bn + col0 + b;
              const int feat = m_tile * kBM + a;
              int row = tok;
              if (e.xg_mask_rows) {
                const int i = tok % e.rows_per_seq;
                row = i == 0 ? -1 : (tok / e.rows_per_seq) * e.gamma + i - 1;
              }
              if (row >= 0) {
                const size_t xi = static_cast<size_t>(row) * e.d_model + feat;
                const float xv = gx * hn;
                if (e.xg_bf16)
                  store_hilo(reinterpret_cast<__nv_bfloat16*>(e.xg_out), xi, e.lo_off, xv);
                else
                  reinterpret_cast<float*>(e.xg_out)[xi] = xv;
              }
              const_cast<float*>(S)[b * kSLD + a] = hn * hn;
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < kB; ++u)
            if (ok[u]) store_out(e.out, e.out_bf16, o[u], v[u]);
        }
      }
      if (kOp == EPI_ADD_F32 && e.xg_out != nullptr) {
        // per token: sum of h_new^2 over the tile's 128 features (fixed order:
        // four strided partials per lane, then a shuffle tree)
        named_bar(1, 128);
        const int w = etid >> 5, lane = etid & 31;
        for (int b = w; b < cols; b += 4) {
          const int tok = n_tile * g.bn + col0 + b;
          float sacc = 0.f;
          for (int i = 0; i < 4; ++i) {
            const int a = lane + 32 * i;
            if (tok < e.n_tok && m_tile * kBM + a < e.n_feat) sacc += S[b * kSLD + a];
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) sacc += __shfl_xor_sync(0xffffffffu, sacc, off);
          int row = tok;
          if (e.xg_mask_rows) {
            const int i = tok % e.rows_per_seq;
            row = i == 0 ? -1 : (tok / e.rows_per_seq) * e.gamma + i - 1;
          }
          if (lane == 0 && tok < e.n_tok && row >= 0)
            e.ss_out[static_cast<size_t>(row) * e.n_ss + m_tile] = sacc;
        }
      }
      if (kOp == EPI_FUSE) {
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
      // A rows 0..63: gate features m_tile*64 + a; rows 64..127: matching up
      // rows. Four consecutive features per thread (16 threads per token),
      // written as one 8-byte (bf16) or 16-byte (fp32) store where aligned.
      const int f0 = m_tile * 64;
      const bool vec = (e.ld % 4) == 0 && (e.lo_off % 4) == 0;
      for (int idx = etid; idx < cols * 16; idx += 128) {
        const int a0 = (idx & 15) * 4, b = idx >> 4;
        const int tok = n_tile * g.bn + col0 + b;
        const int feat = f0 + a0;
        if (tok >= e.n_tok || feat >= e.n_feat) continue;
        const float rs = e.ss_in != nullptr ? rstd[b] : 1.f;
        float y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float gate = S[b * kSLD + a0 + i] * rs, up = S[b * kSLD + a0 + i + 64] * rs;
          y[i] = silu_f(gate) * up;
        }
        const size_t oi = static_cast<size_t>(tok) * e.ld + feat;
        if (vec && feat + 4 <= e.n_feat) {
          if (e.out_bf16) {
            __nv_bfloat16 hi[4], lo[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              hi[i] = __float2bfloat16_rn(y[i]);
              lo[i] = __float2bfloat16_rn(y[i] - __bfloat162float(hi[i]));
            }
            __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(e.out);
            *reinterpret_cast<uint2*>(o + oi) = *reinterpret_cast<const uint2*>(hi);
            if (e.lo_off) *reinterpret_cast<uint2*>(o + oi + e.lo_off) = *reinterpret_cast<const uint2*>(lo);
          } else {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(e.out) + oi) = make_float4(y[0], y[1], y[2], y[3]);
          }
        } else {
          for (int i = 0; i < 4 && feat + i < e.n_feat; ++i) {
            if (e.out_bf16)
              store_hilo(reinterpret_cast<__nv_bfloat16*>(e.out), oi + i, e.lo_off, y[i]);
            else
              reinterpret_cast<float*>(e.out)[oi + i] = y[i];
          }
        }
      }
      break;
    }
    case EPI_QKV:
    case EPI_KV: {
      const int Dh = e.head_dim, half = Dh >> 1;
      const int nq = e.n_q_heads * Dh, nk = e.n_kv_heads * Dh;
      constexpr int kB = epi_batch<kOp, kWide>();
      if constexpr (kWide) {
        // Wide tiles (decode tiles: weights along A rows; a token-major
        // injection takes the direct epilogue): this thread's output feature, its kind (q, k or v),
        // head, RoPE partner row and table column are fixed; its tokens come
        // in batches of 8 whose table loads are all issued first.
        const int a = etid, gf = m_tile * kBM + a;
        int f = gf, layer = e.layer;
        if (kOp == EPI_KV) {
          layer = gf / e.feat_per_layer;
          f = gf - layer * e.feat_per_layer + nq;   // position within the [Q; K; V] rows
        }
        const bool fok = gf < e.n_feat;
        const int d = f % Dh, j = d < half ? d : d - half;
        const int kind = f < nq ? 1 : (f < nq + nk ? 2 : 3);
        const int head = kind == 2 ? (f - nq) / Dh : (f - nq - nk) / Dh;
        const int pa = d < half ? a + half : a - half;   // partner row, same head (in range: 128 % Dh == 0)
        const bool rope = kind != 3 && e.rope_cos != nullptr;
        void* dst = kind == 1 ? e.out : (kind == 2 ? e.k_cache : e.v_cache);
        constexpr int NB = 8;
        for (int b0 = 0; b0 < cols; b0 += NB) {
          float y[NB], p[NB], c[NB], sn[NB];
          int pp[NB];
          bool ok[NB];
#pragma unroll
          for (int u = 0; u < NB; ++u) {
            const int b = b0 + u, tok = n_tile * g.bn + col0 + b;
            const int pos = b < cols ? ti->pos[b] : -1;
            ok[u] = fok && b < cols && (kind == 1 ? tok < e.n_tok : pos >= 0);
            pp[u] = pos < 0 ? 0 : pos;
            y[u] = ok[u] ? S[b * kSLD + a] : 0.f;
            p[u] = ok[u] && rope ? S[b * kSLD + pa] : 0.f;
            c[u] = 1.f;
            sn[u] = 0.f;
            if (ok[u] && rope) {
              const size_t t = static_cast<size_t>(pp[u]) * half + j;
              c[u] = e.rope_cos[t];
              sn[u] = e.rope_sin[t];
            }
          }
#pragma unroll
          for (int u = 0; u < NB; ++u) {
            if (!ok[u]) continue;
            const int b = b0 + u, tok = n_tile * g.bn + col0 + b;
            float val = y[u];
            if (rope) val = d < half ? y[u] * c[u] - p[u] * sn[u] : y[u] * c[u] + p[u] * sn[u];
            if (e.ss_in != nullptr) val *= rstd[b];
            size_t o;
            if (kind == 1) {
              o = static_cast<size_t>(tok) * e.ld + f;
            } else {
              const int sq = ti->seq[b];   // the sequence, or for paged caches the row's page
              o = e.page_table != nullptr
                      ? (((static_cast<size_t>(layer) * e.n_pages + sq) * e.n_kv_heads + head) * kPageKeys +
                         pp[u] % kPageKeys) * Dh + d
                      : (((static_cast<size_t>(layer) * e.max_batch + sq) * e.n_kv_heads + head) * e.ncap + pp[u]) *
                                Dh + d;
            }
            store_out(dst, e.out_bf16, o, val);
          }
        }
      } else {
      for (int base = etid; base < total; base += 128 * kB) {
        float y[kB], cs[kB];  // value and its RoPE partner
        size_t o[kB];
        int kind[kB];  // 0 skip, 1 q, 2 k, 3 v
        int dd[kB], pp[kB], xx[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          const int idx = base + u * 128;
          int a, b;
          if (g.swap) { a = idx & 127; b = idx >> 7; } else { b = idx % cols; a = idx / cols; }
          const int gf = g.swap ? m_tile * kBM + a : n_tile * g.bn + col0 + b;
          const int x = tok_cols ? b : a;
          const int tok = tok_cols ? n_tile * g.bn + col0 + b : m_tile * kBM + a;
          kind[u] = 0;
          dd[u] = 0;
          pp[u] = 0;
          xx[u] = x;
          o[u] = 0;
          y[u] = 0.f;
          if (idx < total && gf < e.n_feat) {
            const int pos = ti->pos[x], seq = ti->seq[x];
            int f = gf, layer = e.layer;
            if (kOp == EPI_KV) {
              layer = gf / e.feat_per_layer;
              f = gf - layer * e.feat_per_layer + nq;   // position within the [Q; K; V] rows
            }
            const int d = f % Dh;
            if (f < nq) {
              kind[u] = 1;
              o[u] = static_cast<size_t>(tok) * e.ld + f;
            } else if (pos >= 0) {
              const bool is_k = f < nq + nk;
              const int head = (is_k ? f - nq : f - nq - nk) / Dh;
              kind[u] = is_k ? 2 : 3;
              // seq: the sequence, or for paged caches the row's page
              o[u] = e.page_table != nullptr
                         ? (((static_cast<size_t>(layer) * e.n_pages + seq) * e.n_kv_heads + head) * kPageKeys +
                            pos % kPageKeys) * Dh + d
                         : (((static_cast<size_t>(layer) * e.max_batch + seq) * e.n_kv_heads + head) * e.ncap + pos) *
                                   Dh + d;
            }
            if (kind[u] == 1 && tok >= e.n_tok) kind[u] = 0;
            if (kind[u] != 0) {
              dd[u] = d;
              pp[u] = pos < 0 ? 0 : pos;
              y[u] = S[b * kSLD + a];
              if (kind[u] != 3 && e.rope_cos != nullptr) {
                const int pa = g.swap ? (d < half ? a + half : a - half) : a;
                const int pb = g.swap ? b : (d < half ? b + half : b - half);
                if (pa < 0 || pa >= kBM || pb < 0 || pb >= cols) {
                  // the RoPE partner lies outside the staged chunk: a head
                  // split across chunks, which the launcher refuses
                  report(g.dev_status, DFLASH_ERR_SHAPE);
                  kind[u] = 0;
                } else {
                  cs[u] = S[pb * kSLD + pa];   // partner value, rotated below
                }
              }
            }
          }
        }
        // table loads of the whole batch first, then the rotations and stores
        float c[kB], sv[kB];
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          c[u] = 1.f;
          sv[u] = 0.f;
          if (kind[u] != 0 && kind[u] != 3 && e.rope_cos != nullptr) {
            const int j = dd[u] < half ? dd[u] : dd[u] - half;
            const size_t t = static_cast<size_t>(pp[u]) * half + j;
            c[u] = e.rope_cos[t];
            sv[u] = e.rope_sin[t];
          }
        }
#pragma unroll
        for (int u = 0; u < kB; ++u) {
          if (kind[u] == 0) continue;
          float val = y[u];
          if (kind[u] != 3 && e.rope_cos != nullptr)
            val = dd[u] < half ? y[u] * c[u] - cs[u] * sv[u] : y[u] * c[u] + cs[u] * sv[u];
          if (e.ss_in != nullptr) val *= rstd[xx[u]];
          void* dst = kind[u] == 1 ? e.out : (kind[u] == 2 ? e.k_cache : e.v_cache);
          store_out(dst, e.out_bf16, o[u], val);
        }
      }
      }
      break;
    }
    case EPI_ARGMAX: {
      // swap orientation: A rows are vocabulary entries, B rows tokens.
      if (e.out == nullptr && !(e.temperature > 0.f)) {
        // greedy, no logits copy: one thread per token scans the tile's 128
        // vocabulary entries (S rows of consecutive tokens fall in different
        // banks); the max of the packed keys is the same whatever the order,
        // and a token costs no chain of dependent warp shuffles
        const int nf = min(kBM, e.n_feat - m_tile * kBM);
        for (int b = etid; b < cols; b += 128) {
          const int tok = n_tile * g.bn + col0 + b;
          if (tok >= e.n_tok) continue;
          const float rs = e.ss_in != nullptr ? rstd[b] : 1.f;
          const float* srow = S + b * kSLD;
          unsigned long long best = 0ull;
#pragma unroll 8
          for (int a = 0; a < nf; ++a) {
            const unsigned long long key = argmax_key(srow[a] * rs, static_cast<uint32_t>(m_tile * kBM + a));
            best = key > best ? key : best;
          }
          e.keys[static_cast<size_t>(tok) * e.keys_ld + m_tile] = best;
        }
        break;
      }
      const int w = etid >> 5, lane = etid & 31;
      for (int b = w; b < cols; b += 4) {
        const int tok = n_tile * g.bn + col0 + b;
        unsigned long long best = 0ull;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int a = lane + 32 * i;
          const int feat = m_tile * kBM + a;
          if (feat < e.n_feat) {
            const float v = S[b * kSLD + a] * (e.ss_in != nullptr ? rstd[b] : 1.f);
            // sampling: rank by v / T + Gumbel noise (a draw from softmax(v / T))
            const float rank = e.temperature > 0.f && tok < e.n_tok
                                   ? v / e.temperature +
                                         rng_gumbel(e.seed, rng_counter(kStreamDraft, tok % e.gamma, tok / e.gamma,
                                                                        static_cast<uint32_t>(feat)))
                                   : v;
            const unsigned long long key = argmax_key(rank, static_cast<uint32_t>(feat));
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
        // one slot per (tile, token): no other CTA writes it, so no atomics
        // (a shared slot per token took 1187 same-address atomics each)
        if (lane == 0 && tok < e.n_tok) e.keys[static_cast<size_t>(tok) * e.keys_ld + m_tile] = best;
      }
      break;
    }
    default:
      break;
  }
}

// ---------------------------------------------------------------- token-major epilogue
// Tokens along A rows (context fusion and injection of a prefill, plain
// projections): TMEM lane = token, column = output feature, so every thread
// owns one token's row of the accumulator and finishes it alone -- 16
// columns per tcgen05.ld, no staging through shared memory, no barrier. The
// global accesses of a thread are 16 consecutive features (64-byte fp32 or
// 32-byte bf16 vectors), and its loads of a batch (RoPE table rows) are all
// issued before they are used.
template <int kOp>
__host__ __device__ constexpr bool token_major_direct() {
  return kOp == EPI_STORE || kOp == EPI_FUSE || kOp == EPI_KV;
}

__device__ __forceinline__ void store16(void* out, int bf16, size_t idx, const float* v) {
  if (bf16) {
    uint4 w[2];
    uint32_t* u = reinterpret_cast<uint32_t*>(w);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      u[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    uint4* d = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + idx);
    d[0] = w[0];
    d[1] = w[1];
  } else {
    float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + idx);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

__device__ __forceinline__ void store8(void* out, int bf16, size_t idx, const float* v) {
  if (bf16) {
    uint4 w;
    uint32_t* u = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      u[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(out) + idx) = w;
  } else {
    float4* d = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + idx);
    d[0] = make_float4(v[0], v[1], v[2], v[3]);
    d[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

template <int kOp>
__device__ void epilogue_token_major(const GemmArgs& g, uint32_t t_lane, int tok, int n_tile) {
  const Epi& e = g.epi;
  const bool live = tok < e.n_tok;
  const int f0 = n_tile * g.bn;  // first feature of the tile
  if (kOp == EPI_STORE || kOp == EPI_FUSE) {
    // vector stores need whole, 16-element-aligned runs of features
    const bool vec = (e.ld % 16) == 0 && (f0 % 16) == 0;
    float ss = 0.f;
    for (int j = 0; j < g.bn; j += 16) {
      float v[16];
      tmem_ld16(t_lane + j, v);
      tmem_ld_wait();
      const int f = f0 + j;
      if (kOp == EPI_FUSE) {
#pragma unroll
        for (int i = 0; i < 16; ++i) ss += v[i] * v[i];
      }
      if (live) {
        const size_t o = static_cast<size_t>(tok) * e.ld + f;
        if (vec && f + 16 <= e.n_feat) {
          store16(e.out, kOp == EPI_FUSE ? 0 : e.out_bf16, o, v);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (f + i < e.n_feat) store_out(e.out, kOp == EPI_FUSE ? 0 : e.out_bf16, o + i, v[i]);
        }
      }
      if (kOp == EPI_FUSE && ((j + 16) % kBM) == 0) {
        // one slot per 128-feature group, summed in ascending feature order
        if (live && f + 16 <= e.n_feat)
          e.row_ss[static_cast<size_t>(tok) * e.n_ss + (f + 16) / kBM - 1] = ss;
        ss = 0.f;
      }
    }
    return;
  }
  // EPI_KV: feature gf of the tile is [K heads ; V heads] of layer gf / fpl.
  // The tile holds whole 128-feature groups (the launcher checks), so a head
  // and its RoPE partner columns d and d + Dh/2 are in the same tile.
  const int Dh = e.head_dim, half = Dh >> 1;
  const int nk = e.n_kv_heads * Dh;
  int pos = -1, seq = 0;
  if (live) {
    seq = tok / e.rows_per_seq;
    const int t = tok - seq * e.rows_per_seq;
    const int base = e.ctx_len[seq], nn = e.n_new[seq];
    if (t < nn && base + nn <= e.ncap - e.reserve) pos = base + t;
    if (pos >= 0 && e.page_table != nullptr) {
      const int pg = e.page_table[static_cast<size_t>(seq) * e.pages_per_seq + pos / kPageKeys];
      if (pg < 0 || pg >= e.n_pages) {
        report(g.dev_status, DFLASH_ERR_CAPACITY);
        pos = -1;
      } else {
        seq = pg;
      }
    }
  }
  for (int h0 = 0; h0 < g.bn; h0 += Dh) {   // one head of K or V per step
    const int gf = f0 + h0;
    const int layer = gf / e.feat_per_layer;
    const int f = gf - layer * e.feat_per_layer;   // position within [K heads ; V heads]
    const bool is_k = f < nk;
    const int head = (is_k ? f : f - nk) / Dh;
    void* dst = is_k ? e.k_cache : e.v_cache;
    const size_t row = e.page_table != nullptr
                           ? ((static_cast<size_t>(layer) * e.n_pages + seq) * e.n_kv_heads + head) * kPageKeys +
                                 (pos >= 0 ? pos % kPageKeys : 0)
                           : ((static_cast<size_t>(layer) * e.max_batch + seq) * e.n_kv_heads + head) * e.ncap +
                                 (pos >= 0 ? pos : 0);
    const bool write = pos >= 0 && gf < e.n_feat;
    const bool rope = is_k && e.rope_cos != nullptr;
    for (int j0 = 0; j0 < half; j0 += 8) {
      float x[8], y[8];   // features j0.. and their partners half + j0..
      tmem_ld8(t_lane + h0 + j0, x);
      tmem_ld8(t_lane + h0 + half + j0, y);
      float4 cv[2], sv[2];
      if (rope && write) {
        const float4* cp = reinterpret_cast<const float4*>(e.rope_cos + static_cast<size_t>(pos) * half + j0);
        const float4* sp = reinterpret_cast<const float4*>(e.rope_sin + static_cast<size_t>(pos) * half + j0);
        cv[0] = __ldg(cp); cv[1] = __ldg(cp + 1);
        sv[0] = __ldg(sp); sv[1] = __ldg(sp + 1);
      }
      tmem_ld_wait();
      if (!write) continue;
      if (rope) {
        const float c[8] = {cv[0].x, cv[0].y, cv[0].z, cv[0].w, cv[1].x, cv[1].y, cv[1].z, cv[1].w};
        const float sn[8] = {sv[0].x, sv[0].y, sv[0].z, sv[0].w, sv[1].x, sv[1].y, sv[1].z, sv[1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float a = x[i], b = y[i];
          x[i] = a * c[i] - b * sn[i];   // rotate-half: (d, d + Dh/2) pairs
          y[i] = b * c[i] + a * sn[i];
        }
      }
      store8(dst, e.out_bf16, row * Dh + j0, x);
      store8(dst, e.out_bf16, row * Dh + half + j0, y);
    }
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
  int epi_ok;
  TokInfo tok;
};

static_assert(sizeof(SmemHeader) + 1023 <= kSmemHeaderBytes, "shared-memory header allowance");

// Tile (m_tile, n_tile) of grid index t. Decode orientation (A = weights):
// n_tile fastest, so the CTAs that share a weight tile are adjacent in launch
// order and read it from HBM once. Token-major orientation (B = weights):
// groups of group_m (16) token tiles, m fastest inside a group, so the CTAs of a
// wave share a few token tiles and a band of weight tiles instead of
// re-streaming either operand for every tile of the other.
__device__ __forceinline__ void tile_of(const GemmArgs& g, int t, int& m, int& n) {
  if (g.swap || g.group_m <= 0) {
    n = t % g.n_tiles;
    m = t / g.n_tiles;
    return;
  }
  const int per_group = g.group_m * g.n_tiles;
  const int grp = t / per_group, first = grp * g.group_m;
  const int gm = min(g.group_m, g.m_tiles - first);
  const int r = t - grp * per_group;
  m = first + r % gm;
  n = r / gm;
}

// Split-K reduction of this CTA's token columns [cb, cb + cols) of a tile:
// the fp32 partials of the kS splits ([col][row] in each cluster CTA's shared
// memory) summed in ascending split order into S. A thread takes items of 4
// rows of one column; kG = 8 / kS items' remote loads of all splits are
// requested before any is added, so a slice of many columns costs a few
// distributed-shared-memory round trips rather than one per item.
template <int kS>
__device__ __forceinline__ void reduce_split_slice(float* S, uint32_t p_local, int cb, int cols, int etid) {
  constexpr int kG = kMaxSplitK / kS > 0 ? kMaxSplitK / kS : 1;
  const int n_items = cols * (kBM / 4);
  for (int it0 = etid; it0 < n_items; it0 += 128 * kG) {
    float4 v[kG][kS];
#pragma unroll
    for (int gi = 0; gi < kG; ++gi) {
      const int it = it0 + gi * 128;
      const int b = it / (kBM / 4), a = (it % (kBM / 4)) * 4;
      const uint32_t off = static_cast<uint32_t>(((cb + b) * kBM + a) * 4);
#pragma unroll
      for (int sp = 0; sp < kS; ++sp)
        v[gi][sp] = it < n_items ? ld_dsmem_f4(mapa_shared(p_local + off, static_cast<uint32_t>(sp)))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int gi = 0; gi < kG; ++gi) {
      const int it = it0 + gi * 128;
      if (it >= n_items) break;
      const int b = it / (kBM / 4), a = (it % (kBM / 4)) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int sp = 0; sp < kS; ++sp) {
        acc.x += v[gi][sp].x; acc.y += v[gi][sp].y; acc.z += v[gi][sp].z; acc.w += v[gi][sp].w;
      }
      S[b * kSLD + a] = acc.x;
      S[b * kSLD + a + 1] = acc.y;
      S[b * kSLD + a + 2] = acc.z;
      S[b * kSLD + a + 3] = acc.w;
    }
  }
}

// One instantiation per (operand type, split activations, epilogue op), so
// that each launch runs only the code of its own case.
template <bool kTF32, bool kSplit, int kOp, bool kWide>
__global__ void __launch_bounds__(kGemmThreads, 3)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap a_map,
                   const __grid_constant__ CUtensorMap b_map, const GemmArgs g, int stages) {
  extern __shared__ uint8_t smem_raw[];
  SmemHeader* hdr = reinterpret_cast<SmemHeader*>(smem_raw);
  const uint32_t raw_s = smem_u32(smem_raw);
  const uint32_t tiles_s = (raw_s + sizeof(SmemHeader) + 1023u) & ~1023u;
  uint8_t* tiles = smem_raw + (tiles_s - raw_s);

  constexpr int kBK = kTF32 ? 32 : 64;  // 128 bytes of k per row either way
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.y;
  int m_tile, n_tile;
  tile_of(g, blockIdx.x, m_tile, n_tile);
  int issued = 0;  // producer: k-steps whose TMA loads were issued
  const int KT = g.k / kBK;
  const int kt0 = split * g.kt_per_split;
  const int nkt = min(g.kt_per_split, KT - kt0);
  const uint32_t a_bytes = kBM * 128u;
  constexpr bool b_split = kSplit;  // hi and lo rows packed in the tile (g.b_pack each)
  const uint32_t b_tile = static_cast<uint32_t>(g.bn) * 128u;
  const int sub_rows = g.bn / g.n_sub;
  const int box_rows = g.b_box_rows > 0 ? g.b_box_rows : sub_rows;    // rows each B box brings
  // ring stride in shared memory (whole tiles, 1024-byte aligned) and the
  // bytes the TMA loads of one stage actually bring
  const uint32_t stage_stride = a_bytes + b_tile;
  const uint32_t stage_tx = a_bytes + static_cast<uint32_t>(g.n_sub * box_rows) * 128u;
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(g.bn)) tmem_cols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&hdr->full[s]), 1);
      mbar_init(smem_u32(&hdr->empty[s]), 1);
    }
    mbar_init(smem_u32(&hdr->accum), 1);
    hdr->abort_flag = 0;
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
        const uint32_t dst = tiles_s + s * stage_stride;
        const uint32_t bar = smem_u32(&hdr->full[s]);
        if (g.a_gateup > 0) {
          tma_load_3d(dst, &a_map, bar, kt * kBK, a_y, a_z, pol_a);
          tma_load_3d(dst + 64 * 128, &a_map, bar, kt * kBK, a_y + g.a_gateup, a_z, pol_a);
        } else {
          tma_load_3d(dst, &a_map, bar, kt * kBK, a_y, a_z, pol_a);
        }
      };
      auto load_b = [&](int s, int kt) {
        const uint32_t dst = tiles_s + s * stage_stride + a_bytes;
        const uint32_t bar = smem_u32(&hdr->full[s]);
        for (int sub = 0; sub < g.n_sub; ++sub) {
          tma_load_3d(dst + sub * sub_rows * 128, &b_map, bar, kt * kBK, b_y + sub * sub_rows, b_z,
                      pol_b);
        }
      };
      // Weights do not depend on the previous kernel: start streaming them
      // before waiting for it (programmatic dependent launch).
      int n_pre = 0;
      if (g.a_weights) {
        n_pre = min(stages, nkt);
        for (int it = 0; it < n_pre; ++it) {
          mbar_expect_tx(smem_u32(&hdr->full[it]), stage_tx);
          load_a(it, kt0 + it);
        }
      }
      pdl_wait();
      for (int it = 0; it < n_pre; ++it) load_b(it, kt0 + it);
      issued = n_pre;
      for (int it = n_pre; it < nkt; ++it) {
        const int s = it % stages, u = it / stages;
        if (u > 0 && !mbar_wait(smem_u32(&hdr->empty[s]), (u - 1) & 1)) {
          report(g.dev_status, DFLASH_ERR_TIMEOUT);
          atomicExch(&hdr->abort_flag, 1);
          break;
        }
        if (*reinterpret_cast<volatile int*>(&hdr->abort_flag)) break;
        mbar_expect_tx(smem_u32(&hdr->full[s]), stage_tx);
        load_a(s, kt0 + it);
        load_b(s, kt0 + it);
        issued = it + 1;
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
        const uint32_t a_addr = tiles_s + s * stage_stride;
        const uint32_t b_addr = a_addr + a_bytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // 4 x 32 bytes of k per 128-byte row
          const uint64_t adesc = sw128_desc(a_addr + k * 32);
          for (int sub = 0; sub < g.n_sub; ++sub) {
            const uint64_t bdesc = sw128_desc(b_addr + sub * sub_rows * 128 + k * 32);
            const uint32_t acc = (it > 0 || k > 0) ? 1u : 0u;
            if (kTF32) {
              tc_mma_tf32(tmem + sub * sub_rows, adesc, bdesc, idesc, acc);
            } else {
              tc_mma_f16(tmem + sub * sub_rows, adesc, bdesc, idesc, acc);
            }
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
    // folded-norm scales of the tile's tokens, off the critical path
    if (rstd_per_tile(g)) folded_rstd(g.epi, hdr->tok.rstd, n_tile * g.bn, g.bn, etid);
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
    if (ok && token_major_direct<kOp>() && !g.swap && g.splits == 1 && g.epi.ss_in == nullptr) {
      epilogue_token_major<kOp>(g, t_lane, m_tile * kBM + row, n_tile);
    } else if (ok) {
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
          // packed split operands: token j = hi product + lo product (this
          // thread's own row of the staging tile, so no barrier is needed)
          if (b_split)
            for (int j = 0; j < g.b_pack; ++j) S[j * kSLD + row] += S[(g.b_pack + j) * kSLD + row];
          named_bar(1, 128);
          apply_epilogue<kOp, kWide>(g, S, &hdr->tok, c * kBM, cols, m_tile, n_tile, etid);
          named_bar(1, 128);
        }
      } else {
        // split-K: park this CTA's fp32 partial tile in its own shared memory
        // ([col][row], the drained pipeline ring); the cluster reduces it below.
        float* P = reinterpret_cast<float*>(tiles);
        for (int j = 0; j < g.bn; j += 16) {
          float v[16];
          tmem_ld16(t_lane + j, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) P[(j + i) * kBM + row] = v[i];
        }
        if (b_split)
          for (int j = 0; j < g.b_pack; ++j) P[j * kBM + row] += P[(g.b_pack + j) * kBM + row];
      }
    }
    tc_fence_before();
  }
  if (g.splits > 1) {
    // Split-K across the CTAs of this cluster (one cluster per output tile,
    // cluster rank = split). After the barrier every partial is visible;
    // CTA r reduces the token columns [c0, c1) of the tile by reading the
    // partials of all splits through distributed shared memory, in ascending
    // split order, then runs the epilogue on them. A second barrier keeps
    // every partial alive until all peers have read it: each CTA arrives as
    // soon as its reads are done and waits only at the very end, so the
    // epilogue runs while slower peers finish reading. Remote loads are slow
    // to return, so each thread requests every split's value before adding.
    cluster_sync();
    if (warp >= 2) {
      const int etid = threadIdx.x - 64;
      const uint32_t rank = cluster_ctarank();
      const int valid = min(g.bn, g.n_rows - n_tile * g.bn);
      const int per = (valid + g.splits - 1) / g.splits;
      const int c0 = static_cast<int>(rank) * per, c1 = min(valid, c0 + per);
      const uint32_t p_local = tiles_s;
      float* S = reinterpret_cast<float*>(tiles + static_cast<size_t>(g.bn) * kBM * 4);
      const bool ok = hdr->epi_ok != 0;
      bool arrived = false;
      for (int cb = c0; cb < c1; cb += kBM) {
        const int cols = min(kBM, c1 - cb);
        if (ok) {
          switch (g.splits) {
            case 2: reduce_split_slice<2>(S, p_local, cb, cols, etid); break;
            case 3: reduce_split_slice<3>(S, p_local, cb, cols, etid); break;
            case 4: reduce_split_slice<4>(S, p_local, cb, cols, etid); break;
            case 5: reduce_split_slice<5>(S, p_local, cb, cols, etid); break;
            case 6: reduce_split_slice<6>(S, p_local, cb, cols, etid); break;
            case 7: reduce_split_slice<7>(S, p_local, cb, cols, etid); break;
            default: reduce_split_slice<8>(S, p_local, cb, cols, etid); break;
          }
        }
        named_bar(1, 128);
        if (cb + kBM >= c1) {  // the last reads of peer partials are done
          cluster_arrive();
          arrived = true;
        }
        if (ok) apply_epilogue<kOp, kWide>(g, S, &hdr->tok, cb, cols, m_tile, n_tile, etid);
        named_bar(1, 128);
      }
      if (!arrived) cluster_arrive();
    } else {
      cluster_arrive();
    }
    cluster_wait();
  }
  __syncthreads();
  // A CTA that gave up a bounded wait must not exit while TMA loads it issued
  // can still land in its shared memory: the producer waits (bounded again)
  // for the transactions of the last `stages` k-steps it issued. Earlier
  // k-steps of the same stages completed before their stage was refilled.
  if (warp == 0 && lane == 0 && *reinterpret_cast<volatile int*>(&hdr->abort_flag)) {
    for (int it = issued > stages ? issued - stages : 0; it < issued; ++it)
      mbar_wait(smem_u32(&hdr->full[it % stages]), (it / stages) & 1);
  }
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
                   bool weights_a, int bn_cap, bool b_split, bool chained) {
  GemmPlan p{};
  const int bk = 128 / elem_bytes;
  const int KT = k / bk;
  // split activations: one tile holding the hi and the lo rows of every
  // token (two rows per token), for up to 128 tokens
  b_split = b_split && 2 * n_rows <= (bn_cap < 256 ? bn_cap : 256);
  const int n16 = ((b_split ? 2 * n_rows : n_rows) + 15) / 16 * 16;
  const int cap1 = bn_cap < 256 ? bn_cap : 256;
  // Two B tiles of at most 256 rows rather than one tile of up to 512 rows
  // (two MMAs): an accumulator of <= 256 TMEM columns leaves room for a
  // second CTA on the SM, whose main loop then runs while this one's
  // epilogue drains. Decode: two halves of the tokens (the weight tile is
  // read twice, the second time from L2, as the two CTAs are adjacent in
  // launch order); token-major: 256-feature tiles.
  bool one_wide = false;
  if (const char* e = getenv("DFLASH_GEMM_ONE_WIDE_TILE")) one_wide = atoi(e) != 0;   // tuning override
  if (n16 <= cap1) {
    p.bn = n16; p.n_sub = 1; p.n_tiles = 1;
  } else if (n16 <= bn_cap && n16 <= kMaxBN && one_wide) {
    p.bn = (n_rows + 31) / 32 * 32; p.n_sub = 2; p.n_tiles = 1;
  } else if (n16 <= bn_cap && n16 <= kMaxBN && weights_a) {
    p.bn = ((n_rows + 1) / 2 + 15) / 16 * 16; p.n_sub = 1; p.n_tiles = 2;
  } else {
    p.bn = cap1; p.n_sub = 1; p.n_tiles = (n_rows + cap1 - 1) / cap1;
  }
  p.m_tiles = m_tiles;
  p.group_m = 0;
  if (!weights_a) {
    p.group_m = 16;
    if (const char* e = getenv("DFLASH_GEMM_GROUP_M")) p.group_m = atoi(e);   // tuning override
  }
  p.b_split = b_split ? 1 : 0;
  // Resident CTAs per SM follow from the accumulator's TMEM columns (512 per
  // SM): narrow tiles (a few tokens) keep three CTAs per SM with a short
  // ring (3 stages), whose prologues and epilogues then overlap the others'
  // streaming; a 256-column accumulator two CTAs, a 512-column one a single
  // CTA; the ring takes what shared memory that leaves.
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(p.bn)) tmem_cols <<= 1;
  const size_t stage = 16384 + static_cast<size_t>(p.bn) * 128;
  const size_t staging = static_cast<size_t>(p.bn < kBM ? p.bn : kBM) * 129 * 4;
  int target = p.bn <= 128 ? 3 : static_cast<int>(512 / tmem_cols);
  if (const char* e = getenv("DFLASH_GEMM_CTAS")) target = atoi(e);   // tuning override
  if (target < 1) target = 1;
  size_t per_cta = static_cast<size_t>(233472 / target) - 1024;
  if (per_cta > 232448) per_cta = 232448;
  int stages = p.bn <= 128 ? 3 : static_cast<int>((per_cta - kSmemHeaderBytes) / stage);
  // narrow tiles of 65-128 rows in a chain of projections: a 2-stage ring
  // where a third 3-stage CTA would not fit beside two others (the three
  // CTAs keep as many stages in flight per SM as two 3-stage ones, and the
  // next projection's CTAs find room as this one's leave)
  if (chained && p.bn <= 128 && target == 3)
    while (stages > 2 && 3 * (kSmemHeaderBytes + static_cast<size_t>(stages) * stage + 1024) > 233472) --stages;
  if (const char* e = getenv("DFLASH_GEMM_STAGES")) stages = atoi(e);   // tuning override
  if (stages > 16) stages = 16;
  if (stages > KT && KT >= 2) stages = KT;
  if (stages < 2) stages = 2;
  while (static_cast<size_t>(stages) * stage < staging) ++stages;
  while (stages > 2 && kSmemHeaderBytes + static_cast<size_t>(stages) * stage > 232448) --stages;
  p.stages = stages;
  p.smem_bytes = kSmemHeaderBytes + static_cast<size_t>(stages) * stage;
  // resident CTAs per SM: shared memory (228 KB per SM, 1 KB reserved per CTA) and TMEM
  int ctas_per_sm = static_cast<int>(233472 / (p.smem_bytes + 1024));
  if (ctas_per_sm > 4) ctas_per_sm = 4;
  while (ctas_per_sm > 1 && ctas_per_sm * tmem_cols > 512) --ctas_per_sm;
  if (ctas_per_sm < 1) ctas_per_sm = 1;
  int splits = 1;
  if (allow_split) {
    // one wave over the resident slots; clusters hold at most 8 CTAs
    const int tiles = m_tiles * p.n_tiles;
    const int slots = num_sms * ctas_per_sm;
    splits = slots / (tiles > 0 ? tiles : 1);
    if (tiles > slots) {
      // More tiles than resident slots: the last, partial wave runs nearly
      // alone. Split K where that shortens the waves: splits s cost
      // ceil(tiles * s / slots) waves of 1/s the length, plus a reduction
      // (taken as 1/8 of a wave per split step above 1).
      double best = 1e30;
      for (int s = 1; s <= kMaxSplitK && s <= KT / 4; ++s) {
        const double waves = static_cast<double>((tiles * s + slots - 1) / slots);
        const double cost = waves / s * (1.0 + 0.125 * (s - 1));
        if (cost < best - 1e-9) { best = cost; splits = s; }
      }
    }
    if (const char* e = getenv("DFLASH_GEMM_SPLITS")) splits = atoi(e);   // tuning override
    if (splits > KT / 4) splits = KT / 4;
    if (splits > kMaxSplitK) splits = kMaxSplitK;
    if (splits < 1) splits = 1;
    // the partial tile and the reduced column slice must fit in the ring
    const size_t ring = static_cast<size_t>(stages) * stage;
    while (splits > 1) {
      const int per = (p.bn + splits - 1) / splits;
      const size_t need = static_cast<size_t>(p.bn) * kBM * 4 + static_cast<size_t>(per < kBM ? per : kBM) * 129 * 4;
      if (need <= ring) break;
      if (splits < kMaxSplitK && splits < KT / 4) ++splits; else { splits = 1; break; }
    }
  }
  p.kt_per_split = (KT + splits - 1) / splits;
  p.splits = (KT + p.kt_per_split - 1) / p.kt_per_split;
  // without split-K the epilogue drains 128 columns at a time, and a packed
  // tile must pair each token's hi and lo columns inside one drain
  if (b_split && p.splits == 1 && p.bn > kBM)
    return plan_gemm(m_tiles, n_rows, k, elem_bytes, num_sms, allow_split, weights_a, bn_cap, false, chained);
  return p;
}

using GemmKernel = void (*)(const CUtensorMap, const CUtensorMap, const GemmArgs, int);

// the wide instance of op kOp where it has one, else its narrow instance
template <bool kTF32, bool kSplit, int kOp, bool kWide>
constexpr GemmKernel gemm_kernel_of() {
  if constexpr (kWide && has_wide(kOp)) return &gemm_tc_kernel<kTF32, kSplit, kOp, true>;
  else return &gemm_tc_kernel<kTF32, kSplit, kOp, false>;
}
template <bool kTF32, bool kSplit, bool kWide, int... kOps>
struct GemmKernelRow {
  static constexpr GemmKernel fns[sizeof...(kOps)] = {gemm_kernel_of<kTF32, kSplit, kOps, kWide>()...};
};
constexpr int kNumEpiOps = 7;
static_assert(EPI_FUSE == kNumEpiOps - 1, "one kernel per epilogue op");
// [narrow | wide][tf32 | bf16 | bf16 with split activations][epilogue op]
const GemmKernel* const kGemmKernels[2][3] = {
    {GemmKernelRow<true, false, false, 0, 1, 2, 3, 4, 5, 6>::fns,
     GemmKernelRow<false, false, false, 0, 1, 2, 3, 4, 5, 6>::fns,
     GemmKernelRow<false, true, false, 0, 1, 2, 3, 4, 5, 6>::fns},
    {GemmKernelRow<true, false, true, 0, 1, 2, 3, 4, 5, 6>::fns,
     GemmKernelRow<false, false, true, 0, 1, 2, 3, 4, 5, 6>::fns,
     GemmKernelRow<false, true, true, 0, 1, 2, 3, 4, 5, 6>::fns},
};
// Tiles whose epilogue gives every thread many tokens (batches of 4 and more
// sequences, prefill) take the wide instances.
bool wide_tile(const GemmArgs& g) { return g.n_rows >= 64; }

cudaError_t launch_gemm(const CUtensorMap& a_map, const CUtensorMap& b_map, const GemmArgs& args,
                        const GemmPlan& plan, cudaStream_t stream, bool pdl) {
  const bool split = args.b_pack > 0;
  if (args.tf32 && split) return cudaErrorInvalidValue;  // split operands are bf16 only
  if (split != (plan.b_split != 0)) return cudaErrorInvalidValue;  // plan sized the other ring
  if (args.epi.op < 0 || args.epi.op >= kNumEpiOps) return cudaErrorInvalidValue;
  // Tokens along A rows (features along B rows): the epilogue stages 128
  // accumulator columns at a time, so a B tile must hold whole 128-feature
  // groups -- the fusion files its sums of squares per group, and RoPE pairs
  // feature d of a head with d +- Dh/2 inside the staged chunk. Injection
  // tiles must also not straddle two layers' features.
  if (!args.swap && (args.epi.op == EPI_FUSE || args.epi.op == EPI_QKV || args.epi.op == EPI_KV) &&
      plan.bn % kBM != 0)
    return cudaErrorInvalidValue;
  if (!args.swap && args.epi.op == EPI_KV &&
      (args.epi.feat_per_layer % plan.bn != 0 || args.b_tiles_per_z * plan.bn != args.epi.feat_per_layer))
    return cudaErrorInvalidValue;
  const int variant = args.tf32 ? 0 : (split ? 2 : 1);
  const int wide = wide_tile(args) ? 1 : 0;
  const GemmKernel kern = kGemmKernels[wide][variant][args.epi.op];
  static bool configured[2][3][kNumEpiOps][64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  bool& done = configured[wide][variant][args.epi.op][dev & 63];
  if (!done) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.m_tiles * plan.n_tiles, plan.splits, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (plan.splits > 1) {  // one cluster per output tile, spanning its splits
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = plan.splits;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, a_map, b_map, args, plan.stages);
}

}  // namespace dfl
