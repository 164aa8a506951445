// Host-side interfaces shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dflash.h"

namespace dfl {

constexpr int kBM = 128;        // MMA M: rows of the A operand per tile
constexpr int kMaxBN = 512;     // B-operand rows per tile (two MMAs of <= 256)
constexpr int kPageKeys = 128;  // keys per KV-cache page (one attention tile)
constexpr int kGemmThreads = 192;

// Epilogue operations of the projection GEMM.
enum EpiOp : int {
  EPI_STORE = 0,    // out[tok, feat] = acc                      (out dtype: out_bf16)
  EPI_ADD_F32 = 1,  // out[tok, feat] += acc                     (fp32 residual stream)
  EPI_QKV = 2,      // block Q/K/V: RoPE(q) -> q_out; RoPE(k), v -> KV cache scratch rows
  EPI_KV = 3,       // injected context K/V: RoPE(k), v -> KV cache at ctx_len + t
  EPI_SWIGLU = 4,   // A tile = 64 gate rows + 64 up rows: out = silu(gate) * up
  EPI_ARGMAX = 5,   // per token: packed (value, index) max -> keys (+ optional fp32 logits)
  EPI_FUSE = 6      // context fusion: u -> out (cfg dtype) and per-row sums of squares
};

struct Epi {
  int op;
  void* out;          // EPI_STORE / EPI_ADD_F32 / EPI_SWIGLU / EPI_FUSE / EPI_QKV (q)
  int ld;             // leading dimension of out (elements)
  int out_bf16;       // 1: out (and caches) are bf16, 0: fp32
  int n_tok;          // valid token rows
  int n_feat;         // valid features
  // attention-layout fields (EPI_QKV / EPI_KV)
  void* k_cache;
  void* v_cache;
  const int* ctx_len;
  const int* n_new;   // EPI_KV: rows per sequence; NULL for EPI_QKV
  int rows_per_seq;   // R for EPI_QKV, Tmax for EPI_KV
  int layer;          // EPI_QKV: layer; EPI_KV: layer of feature tile 0 (see feat_per_layer)
  int feat_per_layer; // EPI_KV: 2*Hkv*Dh features per layer (layer = feat / feat_per_layer)
  int max_batch, n_q_heads, n_kv_heads, head_dim, ncap, reserve;
  // paged caches (page_table != NULL): k_cache / v_cache are page pools
  // [L][n_pages][Hkv][kPageKeys][Dh]; key p of sequence s lives in page
  // page_table[s * pages_per_seq + p / kPageKeys], row p % kPageKeys; ncap is
  // then pages_per_seq * kPageKeys
  const int32_t* page_table;
  int n_pages, pages_per_seq;
  const float* rope_cos;
  const float* rope_sin;
  int rope_positions;
  // EPI_ARGMAX: keys[tok * keys_ld + m_tile] = packed (value, index) max of
  // token tok over the tile's 128 vocabulary entries (every entry written)
  unsigned long long* keys;
  int keys_ld;
  // EPI_ARGMAX sampling mode (temperature > 0): token t = b * gamma + j ranks
  // vocabulary entry v by logit / temperature + Gumbel(seed, stream 0, j, b, v)
  float temperature;
  uint64_t seed;
  // EPI_FUSE
  float* row_ss;      // [n_tok, n_ss] partial sums of squares
  int n_ss;
  // RMSNorm folded into the projections. Consumer side: when ss_in is set,
  // the accumulator of token t is scaled by rstd[t] = 1/sqrt(sum(ss_in[t]) / d_model + eps)
  // (its B operand is g (.) h, so the product equals W RMSNorm(h)).
  // Producer side (EPI_ADD_F32): when xg_out is set, also writes
  // xg_out[row] = g (.) h_new (cfg dtype) and ss_out[row][m_tile] = sum over
  // the tile's 128 features of h_new^2; xg_mask_rows maps token b*R + i to
  // row b*gamma + i - 1 and skips the anchor rows (the final norm's rows).
  const float* ss_in;
  void* xg_out;
  const void* xg_gain;
  float* ss_out;
  int xg_mask_rows;
  int xg_bf16;        // element type of xg_out and xg_gain
  size_t lo_off;      // > 0: bf16 outputs feeding a projection (xg_out, or out of
                      // EPI_SWIGLU) also get lo = bf16(x - hi) at + lo_off elements
  int gamma;
  int d_model;
  float eps;
};

struct GemmArgs {
  int m_rows;         // valid rows of the A operand
  int n_rows;         // valid rows of the B operand
  int k;              // reduction length in elements
  int bn;             // B rows per tile (multiple of 16 per MMA)
  int n_sub;          // MMAs per k-step (bn / n_sub rows each)
  int kt_per_split;   // k-tiles per split
  int splits;
  int m_tiles, n_tiles;
  // TMA coordinates: row = row0 + (tile % tiles_per_z) * tile_rows, z = z0 + tile / tiles_per_z
  int a_row0, a_z0, a_tiles_per_z;
  int b_row0, b_z0, b_tiles_per_z;
  int a_gateup;       // > 0: A tile = 64 rows at a_row0 + 64*m and 64 rows at a_row0 + a_gateup + 64*m
  int b_pack;         // > 0: split activations packed in one B tile: rows [0, b_pack) hold
                      //      hi = bf16(x) and rows [b_pack, 2 b_pack) lo = bf16(x - hi) of
                      //      the same tokens; accumulator column b_pack + j is added to column j
  int b_box_rows;     // rows per B box of the tensor map (0: bn / n_sub); rows of a tile
                      // past the box are never loaded and feed only unused accumulator columns
  int swap;           // 1: A rows are output features and B rows tokens; 0: the reverse
  int group_m;        // token-major tiles: grid order in groups of group_m A tiles (0: n fastest)
  int a_weights;      // 1: A is a weight (independent of earlier kernels): prefetch before PDL wait
  int tf32;           // 1: fp32 operands through kind::tf32
  int* dev_status;
  Epi epi;
};

struct GemmPlan {
  int bn, n_sub, splits, kt_per_split, m_tiles, n_tiles, stages;
  int group_m;        // grid order (GemmArgs::group_m)
  int b_split;        // B tile packs hi and lo rows (bn covers 2 n_rows)
  size_t smem_bytes;
};

// Chooses tile shape, split count, pipeline depth and grid order for
// m_tiles A tiles against n_rows B rows over k (elements of elem_bytes each);
// weights_a: A is the weight matrix (decode orientation), else B is.
// chained: one of the drafting pass's back-to-back projections (each hands
// its SMs to the next through programmatic dependent launch).
GemmPlan plan_gemm(int m_tiles, int n_rows, int k, int elem_bytes, int num_sms, bool allow_split,
                   bool weights_a, int bn_cap = kMaxBN, bool b_split = false, bool chained = false);

// Builds a 3-D tensor map over a [z][rows][k] row-major operand with a box of
// (64 or 32 elements of k) x box_rows x 1 and 128-byte swizzle.
bool make_operand_map(CUtensorMap* map, const void* base, int elem_bytes, uint64_t k,
                      uint64_t rows, uint64_t zdim, uint32_t box_rows);

cudaError_t launch_gemm(const CUtensorMap& a_map, const CUtensorMap& b_map, const GemmArgs& args,
                        const GemmPlan& plan, cudaStream_t stream, bool pdl);

// Attention over [injected context ; block] for one layer.
struct AttnArgs {
  const void* q;          // [B*R, Hq*Dh]
  const void* k_cache;    // whole cache [L, max_batch, Hkv, Ncap, Dh]
  const void* v_cache;
  int layer, n_layers;
  const int* ctx_len;     // [B]
  const int* gamma_b;     // NULL or [B]: block of sequence b is rows 0..gamma_b[b] (keys
                          // ctx_len[b] + gamma_b[b] + 1); rows past it are inert
  void* out;              // [B*R, Hq*Dh]
  size_t out_lo_off;      // > 0: bf16 lo = bf16(o - hi) at out + out_lo_off elements
  int* dev_status;
  int B, R, n_q_heads, n_kv_heads, head_dim, ncap, max_batch;
  int splits, chunk;      // keys per split of the longest context (multiple of 128); the
                          // tcgen05 kernel splits each sequence's own keys evenly (whole
                          // 128-key tiles); the last split takes the rest
  int merge_global;       // 0: the splits of one (sequence, KV head) form one cluster and merge
                          //    through distributed shared memory;
                          // 1: more splits than a cluster holds: each writes its partial rows
                          //    to `partials` and a second kernel merges them
  float* partials;        // merge_global: [B][Hkv][splits] slots of attn_slot_floats(head_dim)
  int bf16;
  const int32_t* page_table;   // NULL, or paged caches as in Epi
  int n_pages, pages_per_seq;
  int prefetch_tiles;          // K/V tiles per split asked of L2 before the dependency wait
};
// Floats of one split's partial result: 128 unnormalised O rows of head_dim,
// then (running max, row sum) of each row.
__host__ __device__ constexpr size_t attn_slot_floats(int head_dim) {
  return static_cast<size_t>(128) * head_dim + 256;
}
// Partial-result slots in a workspace: B * Hkv * splits on the merge_global path.
constexpr int kAttnMaxSlots = 160;
// Split-KV plan for B sequences over at most max_ctx context keys on a device
// with num_sms SMs.
void plan_attention(int B, int R, int Hq, int Hkv, int Dh, int max_ctx, int ncap, int num_sms,
                    int* splits, int* chunk, int* merge_global);
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream, bool pdl);
// bf16 path on tcgen05 (attention_tc.cu)
cudaError_t launch_attention_tc(const AttnArgs& a, cudaStream_t stream, bool pdl);
// Second kernel of the merge_global path (a no-op launch otherwise).
cudaError_t launch_attention_merge(const AttnArgs& a, cudaStream_t stream, bool pdl);

// Small row kernels.
// h[b*R + i] = embed[id] (id = ids[b*R + i] when ids is given, else anchor[b]
// for i == 0 and mask_id otherwise), fp32; also xg = gain (.) h in cfg dtype
// and ss[row][c] = sum of h^2 over features 128c..128c+127 (the first
// layer's folded RMSNorm).
cudaError_t launch_embed(const void* embed, const int* anchor, const int* ids, int mask_id, int B, int R,
                         int D, int V,
                         int bf16, float* h, const void* gain, void* xg, size_t xg_lo_off, float* ss,
                         int* dev_status, cudaStream_t s, bool pdl);
// h[t] = gain * u[t] / sqrt(sum(row_ss[t]) / D + eps), u fp32, h in cfg dtype.
cudaError_t launch_fuse_norm(const float* u, void* h, const float* row_ss, int n_ss, const void* gain,
                             int T, int D, float eps, int bf16, cudaStream_t s, bool pdl);
// Multi-step confidence unmasking (unmask.cu). ids [B, R] block inputs.
cudaError_t launch_ids_init(const int32_t* anchor, int mask_id, int B, int R, int32_t* ids, cudaStream_t s,
                            bool pdl);
// One unmasking decision per sequence from the pass's logits [B, gamma, V]
// (fp32) and argmax tokens draft [B, gamma]: the ceil(m / steps_left) most
// confident still-masked positions take their token. ws: sample_ws_bytes.
cudaError_t launch_unmask_step(const float* logits, const int32_t* draft, int B, int gamma, int V,
                               int mask_id, int steps_left, void* ws, int32_t* ids, cudaStream_t s,
                               bool pdl);
cudaError_t launch_ids_to_draft(const int32_t* ids, int B, int gamma, int32_t* draft, cudaStream_t s,
                                bool pdl);

// Sampling verification (temperature > 0): rejection-acceptance over the
// target logits [B, gamma+1, V] (bf16 or fp32) and the drafter logits
// [B, gamma, V] (fp32) of the sampled drafts. Three launches: per-chunk
// softmax statistics of every row, the acceptance scan (one CTA per
// sequence), and the residual / bonus draw over V with the decision.
constexpr int kSampChunk = 4096;  // vocabulary entries per statistics CTA
struct SampleState {
  int a;                 // accepted drafts
  float mt, st, md, sd;  // softmax max and sum (of logit / T) of target and draft row a
  int pad[3];
};
size_t sample_ws_bytes(int max_batch, int gamma, int vocab);
cudaError_t launch_sample_verify(const void* target, int target_bf16, const float* draft_logits,
                                 const int32_t* draft, int B, int gamma, int V, float temperature,
                                 uint64_t seed, void* ws, int32_t* tau, int32_t* committed,
                                 int32_t* next_anchor, cudaStream_t s, bool pdl);
// draft[t] = index of the max of keys[t * ld + 0 .. n_tiles) (the LM head's
// per-tile maxima); with gamma_b, t = b * gamma + j with j >= gamma_b[b] gets -1.
cudaError_t launch_argmax_finalize(const unsigned long long* keys, int n_tiles, int ld, int n, int gamma,
                                   const int32_t* gamma_b, int32_t* draft, cudaStream_t s, bool pdl);
cudaError_t launch_kv_advance(int32_t* ctx_len, const int32_t* n_new, int B, int Tmax, int ncap,
                              int reserve, int* dev_status, cudaStream_t s, bool pdl);
// Greedy verify-accept; gamma_b NULL or [B] (sequence b verifies its first gamma_b[b] drafts).
cudaError_t launch_verify(const void* logits, int bf16, const int32_t* draft, const int32_t* gamma_b,
                          int B, int gamma, int V, int32_t* tau, int32_t* committed,
                          int32_t* next_anchor, unsigned long long* keys, int* counters,
                          cudaStream_t s, bool pdl);
cudaError_t launch_copy_f32(float* dst, const float* src, size_t n, cudaStream_t s, bool pdl);
// One CTA whose bounded wait on an mbarrier nothing arrives on runs out.
cudaError_t launch_wait_selftest(int* dev_status, cudaStream_t s);

int num_sms_of_current_device();
// DFLASH_ERR_ARCH unless the current device is sm_103 (cached per device).
dflash_status check_arch();
// Programmatic dependent launch on (default) unless DFLASH_PDL=0.
bool use_pdl();
// V-chunks per target row of verify_kernel: about two CTAs per SM in total.
int verify_chunks(int B, int R, int V, int num_sms);

}  // namespace dfl
