/*
 * dflash.h -- C ABI of the GB300-native DFlash drafting step.
 *
 * DFlash drafts a whole block of tokens in one forward pass of a small
 * block-diffusion drafter whose every layer attends to K/V projected from a
 * fused feature of the target model's hidden states ("KV injection").
 *
 * Sources (cited by page title and section throughout this library):
 *   [P1] "DFlash: Block Diffusion for Flash Speculative Decoding 논문 정리"
 *        (juhoplayground.github.io): sections "Preliminaries" (eq. (1)),
 *        "추론 구조" (inference structure), "KV Injection 메커니즘".
 *   [P2] "DFlash 블록 확산 디코딩: 투기적 디코딩의 드래프트 비용을 상수로 만드는 법"
 *        (blog.gillilab.com): sections on speculative drafting and cost.
 *   [P4] "ICML'26 | DFlash：用 Diffusion 模型干掉 AR Drafter，投机解码提速 6×"
 *        (marsggbo.github.io): §3.1 context feature, §3.2 KV injection,
 *        §3.3 one-pass block prediction.
 *
 * Conventions shared by every entry point:
 *  - All tensor arguments are DEVICE pointers to caller-owned, contiguous,
 *    row-major memory unless the comment says "host". The library allocates
 *    no device memory; scratch comes from the caller's workspace `ws`.
 *  - Every call is asynchronous on `stream` and never synchronises. Nothing
 *    is launched when a call returns a non-OK status.
 *  - Host-detectable errors (null pointers, bad shapes, too small workspace,
 *    wrong device architecture) are returned as a negative dflash_status.
 *    Device-detected errors (cache capacity overflow, a bounded wait that
 *    ran out) are written to the int32 `dev_status` word (first error wins,
 *    the offending write is skipped); it must be 0 before the call.
 *  - Token ids are int32. The block has R = gamma + 1 rows: the anchor
 *    followed by gamma mask tokens ([P4] §3.3). gamma <= DFLASH_MAX_GAMMA.
 *  - Stacked per-layer weights: tensor kind X of layer l starts at
 *    X + l * (rows * cols) elements.
 *  - Element type of weights, taps, hidden states and KV cache is cfg.dtype
 *    (bf16 or fp32). Residual-stream arithmetic, softmax and all
 *    accumulation are fp32 on the GPU.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_ABI_VERSION 1
#define DFLASH_MAX_GAMMA 16

/* Same object as cudaStream_t / CUstream; declared here so that this header
 * needs no CUDA include. NULL means the legacy default stream. */
typedef struct CUstream_st* dflash_stream_t;

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = -1, /* null pointer or out-of-range scalar        */
  DFLASH_ERR_SHAPE = -2,       /* unsupported model shape                      */
  DFLASH_ERR_DTYPE = -3,       /* unsupported element type                     */
  DFLASH_ERR_CAPACITY = -4,    /* KV cache too small (device side: dev_status) */
  DFLASH_ERR_ARCH = -5,        /* current device is not sm_103                 */
  DFLASH_ERR_CUDA = -6,        /* a CUDA runtime/driver call failed            */
  DFLASH_ERR_TIMEOUT = -7,     /* device: a bounded wait ran out               */
  DFLASH_ERR_WORKSPACE = -8,   /* workspace missing or too small               */
  DFLASH_ERR_ALIGN = -9,       /* pointer not 16-byte aligned                  */
  DFLASH_ERR_TOO_LARGE = -10   /* request beyond a fixed maximum size          */
} dflash_status;

typedef enum { DFLASH_F32 = 0, DFLASH_BF16 = 1 } dflash_dtype;

/* Model and capacity description (plain data, copied by value on each call). */
typedef struct {
  int n_layers;      /* L drafter layers ([P1] 실험 설정: 5, or 8)             */
  int d_target;      /* Dt, target hidden size                                 */
  int n_taps;        /* tapped target layers concatenated ([P1]: 5)            */
  int d_model;       /* D, drafter hidden size                                 */
  int n_q_heads;     /* Hq                                                     */
  int n_kv_heads;    /* Hkv (Hq % Hkv == 0; q head h reads kv head h/(Hq/Hkv)) */
  int head_dim;      /* Dh: 64 or 128                                          */
  int d_ffn;         /* F, SwiGLU width                                        */
  int vocab;         /* V                                                      */
  int gamma;         /* number of mask tokens drafted per block (1..16)        */
  int mask_token_id; /* id fed at the gamma mask positions                    */
  int max_batch;     /* batch stride of the KV cache                           */
  int ctx_capacity;  /* Ncap: KV-cache rows per (layer, sequence, kv head)     */
  float rms_eps;     /* RMSNorm epsilon                                        */
  float rope_theta;  /* RoPE base; 0 disables rotary position encoding         */
  dflash_dtype dtype;
} dflash_config;

/* Drafter parameters: caller-owned DEVICE pointers, element type cfg.dtype
 * (rope tables are fp32). Row-major [out, in] like a linear layer. */
typedef struct {
  const void* w_c;       /* [D, n_taps*Dt]   context fusion W_c               */
  const void* g_c;       /* [D]              its RMSNorm gain                 */
  const void* embed;     /* [V, D]           token embedding                  */
  const void* g_final;   /* [D]              final RMSNorm gain               */
  const void* lm_head;   /* [V, D]           LM head                          */
  const void* g_attn;    /* [L, D]           pre-attention RMSNorm gains      */
  const void* w_qkv;     /* [L, (Hq+2Hkv)*Dh, D] rows: Q heads, K heads, V heads */
  const void* w_o;       /* [L, D, Hq*Dh]                                     */
  const void* g_ffn;     /* [L, D]           pre-FFN RMSNorm gains            */
  const void* w_gateup;  /* [L, 2F, D]       rows 0..F-1 gate, F..2F-1 up     */
  const void* w_down;    /* [L, D, F]                                         */
  const float* rope_cos; /* [rope_positions, Dh/2]; NULL when rope_theta == 0 */
  const float* rope_sin; /* [rope_positions, Dh/2]                            */
  int rope_positions;    /* rows of the rope tables (> every position used)   */
} dflash_weights;

/* Optional per-launch timing hook. When a call receives a non-NULL trace,
 * it records events[2*i] before and events[2*i+1] after its i-th kernel
 * launch on `stream` (caller-created cudaEvent_t handles, passed as void*),
 * stores the launch's kernel kind in kinds[i] and its algorithmic bytes and
 * flops in bytes[i] / flops[i] (host arrays), and advances *count. Launches
 * beyond `capacity` pairs are not traced. Tracing serialises launches, so a
 * traced run is for attribution, not for the headline time. */
typedef enum {
  DFLASH_K_GEMM = 0,      /* tcgen05 projection GEMM (all epilogues)      */
  DFLASH_K_ATTN = 1,      /* split-KV context attention + merge           */
  DFLASH_K_NORM = 2,      /* RMSNorm / embedding / small row kernels      */
  DFLASH_K_ARGMAX = 3,    /* argmax finalisation                          */
  DFLASH_K_VERIFY = 4     /* verify-accept                                */
} dflash_kernel_kind;

typedef struct {
  void** events;   /* host array of 2*capacity cudaEvent_t           */
  int capacity;
  int count;       /* in/out: launches traced so far                  */
  int* kinds;      /* host [capacity]                                 */
  double* bytes;   /* host [capacity] algorithmic HBM bytes per launch */
  double* flops;   /* host [capacity] algorithmic flops per launch     */
} dflash_trace;

/* Paged KV cache (a ragged layout for serving-style continuous batching,
 * without padding every sequence to one capacity; the pages describe the
 * cache only as computed once per position and reused, [P1] "추론 구조"). Each layer's K
 * and V live in a pool of pages of DFLASH_PAGE_KEYS positions:
 *   pool[L][n_pages][Hkv][DFLASH_PAGE_KEYS][Dh]  (cfg.dtype)
 * and position p of sequence b in page page_table[b * pages_per_seq + p /
 * DFLASH_PAGE_KEYS], row p % DFLASH_PAGE_KEYS. A sequence's capacity is
 * pages_per_seq * DFLASH_PAGE_KEYS positions (replacing cfg.ctx_capacity for
 * the *_paged calls; the last gamma + 1 of them are the draft block's
 * scratch rows, as in the contiguous cache). The caller owns the pools and
 * the table and allocates pages before positions reach them; a write or
 * read through an entry outside [0, n_pages) sets DFLASH_ERR_CAPACITY in
 * dev_status (writes are skipped). Every page covers one 128-key attention
 * tile, so a tile is a single TMA box wherever the page sits in the pool. */
#define DFLASH_PAGE_KEYS 128
typedef struct {
  void* k_pool;               /* device [L, n_pages, Hkv, DFLASH_PAGE_KEYS, Dh] */
  void* v_pool;               /* device, same shape                              */
  const int32_t* page_table;  /* device [max_batch, pages_per_seq] page ids      */
  int n_pages;                /* pages in each pool                              */
  int pages_per_seq;          /* table entries per sequence                      */
} dflash_kv_pages;

/* ABI version compiled into the library (DFLASH_ABI_VERSION). */
int dflash_abi_version(void);

/* Static string naming a status code. Never NULL. */
const char* dflash_status_string(dflash_status s);

/* Checks a configuration without touching the GPU. Returns DFLASH_OK or the
 * first violated constraint (DFLASH_ERR_SHAPE / _DTYPE / _INVALID_ARG). */
dflash_status dflash_check_config(const dflash_config* cfg);

/* Bytes of one stacked parameter set for cfg (host arithmetic only).
 * kind: 0 = W_c, 1 = embedding, 2 = LM head, 3 = all L layers (QKV, O,
 * gate|up, down, two gains), 4 = total. Returns 0 on a bad cfg/kind. */
size_t dflash_param_bytes(const dflash_config* cfg, int kind);

/* Bytes of one KV cache tensor (K or V): L * max_batch * Hkv * Ncap * Dh
 * elements of cfg.dtype. */
size_t dflash_kv_cache_bytes(const dflash_config* cfg);

/* Workspace bytes needed by every call below for up to `max_rows` token
 * rows per dflash_ctx_fuse / dflash_kv_inject call (T, or B*Tmax) and up to
 * cfg.max_batch sequences per draft / verify call. 0 on a bad cfg. */
size_t dflash_workspace_bytes(const dflash_config* cfg, int max_rows);

/* Failure-detection self-test. Every kernel of this library bounds its waits
 * on mbarriers (about 1 s of SM clock, 2e9 cycles) and, when one runs out,
 * writes DFLASH_ERR_TIMEOUT to the status word and exits instead of hanging.
 * This call launches one CTA whose wait, through the same bounded-wait
 * routine, has nothing to wait for: after about a second dev_status (device
 * int32, 0 before the call) holds DFLASH_ERR_TIMEOUT and the context is still
 * usable. Asynchronous on `stream`. */
dflash_status dflash_selftest_wait_timeout(int32_t* dev_status, dflash_stream_t stream);

/* Zeroes a workspace once after allocation (its tile counters must start at
 * zero; every kernel leaves them at zero again). Asynchronous on stream. */
dflash_status dflash_workspace_init(void* ws, size_t ws_bytes,
                                    dflash_stream_t stream);

/* Context fusion, [P1] "KV Injection 메커니즘" H_t equation and [P4] §3.1:
 *   u_t   = W_c [H(l1)_t ; ... ; H(l5)_t]      (feature-axis concatenation)
 *   H_t   = g_c * u_t / sqrt(mean(u_t^2) + eps)   (RMSNorm over D)
 * taps:  [T, n_taps*Dt] -- row t is the n_taps tapped hidden states of the
 *        same token laid end to end in tap order (l1 first).
 * h_ctx: [T, D] output, cfg.dtype. T >= 0 (T == 0 launches nothing).
 * trace: NULL or a dflash_trace (see above).
 * Errors: DFLASH_ERR_INVALID_ARG for null pointers with T > 0,
 *         DFLASH_ERR_WORKSPACE when T exceeds the workspace's max_rows. */
dflash_status dflash_ctx_fuse(const dflash_config* cfg, const dflash_weights* w,
                              const void* taps, int T, void* h_ctx,
                              void* ws, size_t ws_bytes, dflash_trace* trace,
                              dflash_stream_t stream);

/* KV injection, [P1] "KV Injection 메커니즘" (K_i, V_i equations) and
 * "추론 구조" (cached and reused across drafting iterations):
 *   for every layer i and new context row t of sequence b at absolute
 *   position p = ctx_len[b] + t:
 *     K_cache[i][b][g][p] = RoPE_p(W_i^K H_t)_g ,  V_cache[i][b][g][p] = (W_i^V H_t)_g
 *   then ctx_len[b] += n_new[b] (on the device, after all writes).
 * h_ctx:   [B, Tmax, D]; rows t >= n_new[b] of sequence b are ignored.
 * n_new:   device [B], 0 <= n_new[b] <= Tmax.
 * ctx_len: device [B], advanced in place.
 * k_cache, v_cache: [L, max_batch, Hkv, Ncap, Dh] (cfg.dtype).
 * dev_status: device int32; DFLASH_ERR_CAPACITY when ctx_len[b] + n_new[b]
 *   would exceed Ncap - R (the last R rows are reserved for the draft block);
 *   that sequence is then neither written nor advanced.
 * trace: NULL or a dflash_trace (see above). */
dflash_status dflash_kv_inject(const dflash_config* cfg, const dflash_weights* w,
                               const void* h_ctx, const int32_t* n_new, int B,
                               int Tmax, int32_t* ctx_len, void* k_cache,
                               void* v_cache, int32_t* dev_status, void* ws,
                               size_t ws_bytes, dflash_trace* trace,
                               dflash_stream_t stream);

/* One-pass block drafting, [P4] §3.2-§3.3 and [P1] "추론 구조":
 *   h = Embed([anchor_b, m, ..., m])  (R rows at positions ctx_len[b]+0..gamma)
 *   per layer: a = RMSNorm(h); q,k,v = W_qkv a (RoPE on q and k);
 *     o = softmax(q [K_ctx; k]^T / sqrt(Dh)) [V_ctx; v]  (GQA, bidirectional
 *         inside the block, every row sees all ctx_len[b] + R keys);
 *     h += W_o o;  f = RMSNorm(h);  h += W_down(silu(W_gate f) * W_up f)
 *   z = RMSNorm(h[mask rows]); draft = argmax_V(W_lm z) (lowest index on ties)
 * anchor:  device [B] token ids, 1 <= B <= cfg.max_batch; ctx_len: device [B]
 *   (not modified). A pass of up to 512 block rows (B * (gamma + 1)) runs as
 *   one projection tile of tokens; larger passes take several 256-row tiles.
 * max_ctx_hint: host upper bound of ctx_len[b] used to size the split-KV grid
 *   (any value is correct; a tight one is faster). Must be >= 0. The kernel
 *   divides each sequence's own keys (its device-side ctx_len) among the
 *   splits; a trace record counts an attention launch's K/V bytes and flops
 *   as if every sequence had max_ctx_hint keys.
 * k_cache, v_cache: as in dflash_kv_inject. The block's own K/V rows are
 *   written to cache rows ctx_len[b] .. ctx_len[b]+gamma as scratch; those
 *   rows lie beyond ctx_len and carry no context.
 * draft: device [B, gamma] int32 output.
 * logits_opt: NULL or device fp32 [B, gamma, V] (debug copy of the logits).
 * layer_dump_opt: NULL or device fp32 [L+1, B*R, D]: the residual stream
 *   after the embedding and after each layer.
 * trace: NULL or a dflash_trace (see above). */
dflash_status dflash_draft_block(const dflash_config* cfg, const dflash_weights* w,
                                 const int32_t* anchor, const int32_t* ctx_len,
                                 int B, int max_ctx_hint, void* k_cache,
                                 void* v_cache, int32_t* draft, float* logits_opt,
                                 float* layer_dump_opt, int32_t* dev_status,
                                 void* ws, size_t ws_bytes, dflash_trace* trace,
                                 dflash_stream_t stream);

/* dflash_kv_inject and dflash_draft_block over a paged KV cache
 * (dflash_kv_pages): the same computation, with every cache row addressed
 * through the page table. The RoPE tables must cover the paged capacity.
 * Results equal the contiguous calls' bit for bit. */
dflash_status dflash_kv_inject_paged(const dflash_config* cfg, const dflash_weights* w,
                                     const void* h_ctx, const int32_t* n_new, int B, int Tmax,
                                     int32_t* ctx_len, const dflash_kv_pages* pages,
                                     int32_t* dev_status, void* ws, size_t ws_bytes,
                                     dflash_trace* trace, dflash_stream_t stream);
dflash_status dflash_draft_block_paged(const dflash_config* cfg, const dflash_weights* w,
                                       const int32_t* anchor, const int32_t* ctx_len, int B,
                                       int max_ctx_hint, const dflash_kv_pages* pages,
                                       int32_t* draft, float* logits_opt, int32_t* dev_status,
                                       void* ws, size_t ws_bytes, dflash_trace* trace,
                                       dflash_stream_t stream);

/* Drafting pass with a block size per sequence ([P1] block-size ablation:
 * a drafter trained with block 16 serves smaller inference blocks, which
 * makes per-request block sizes possible;
 * the scheduling policy itself is left to the caller). Sequence b drafts
 * the block [anchor_b, m x gamma_b[b]] at positions ctx_len[b] + 0..gamma_b[b]:
 * exactly dflash_draft_block with gamma = gamma_b[b] for that sequence. Rows
 * past a sequence's block are computed on the padded layout but are neither
 * keys nor drafts: draft[b, j] = -1 for j >= gamma_b[b].
 * gamma_b: device [B] int32, values clamped to [1, cfg.gamma].
 * logits_opt rows j >= gamma_b[b] hold unused values. Other arguments as in
 * dflash_draft_block (no layer dump). */
dflash_status dflash_draft_block_dyn(const dflash_config* cfg, const dflash_weights* w,
                                     const int32_t* anchor, const int32_t* ctx_len,
                                     const int32_t* gamma_b, int B, int max_ctx_hint,
                                     void* k_cache, void* v_cache, int32_t* draft,
                                     float* logits_opt, int32_t* dev_status, void* ws,
                                     size_t ws_bytes, dflash_trace* trace,
                                     dflash_stream_t stream);

/* Greedy verification of blocks of per-sequence size gamma_b[b] (clamped to
 * [1, cfg.gamma]): dflash_verify_accept with gamma = gamma_b[b], reading
 * target rows 0..gamma_b[b] of the [B, gamma+1, V] layout and drafts
 * 0..gamma_b[b]-1 of the [B, gamma] layout; tau[b] in [1, gamma_b[b] + 1];
 * committed[b] is padded with -1 to gamma + 1 entries. */
dflash_status dflash_verify_accept_dyn(const dflash_config* cfg, const void* target_logits,
                                       dflash_dtype logits_dtype, const int32_t* draft,
                                       const int32_t* gamma_b, int B, int32_t* tau,
                                       int32_t* committed, int32_t* next_anchor, void* ws,
                                       size_t ws_bytes, dflash_trace* trace,
                                       dflash_stream_t stream);

/* Multi-step confidence unmasking ([P2] drafting paragraph: the block
 * starts as [MASK] everywhere; each pass predicts all masked positions; the
 * most confident positions are unmasked first; the passes repeat until the
 * block is full). Readings: confidence = max_v softmax(logits_j); pass s of
 * n_steps fills ceil(m / (n_steps - s)) of the m still-masked positions with
 * their argmax tokens, ties to the lower position; filled positions are
 * inputs to later passes.
 *
 * dflash_draft_block_ids: the drafting pass on explicit block inputs
 *   ids [B, R] (device int32; row 0 the anchor, mask_token_id where masked)
 *   instead of [anchor, m, ..., m]; draft = argmax of every mask row's logits.
 * dflash_unmask_step: one decision: logits [B, gamma, V] fp32 and draft
 *   [B, gamma] of the pass on ids; fills the ceil(m / steps_left) most
 *   confident masked positions of ids (in place). steps_left >= 1.
 * dflash_draft_block_iter: n_steps (1..gamma) passes and decisions from
 *   [anchor, m, ..., m]; ids [B, R] receives the final block, draft [B, gamma]
 *   its tokens; logits [B, gamma, V] fp32 is required scratch (it holds the
 *   last pass's logits). n_steps = 1 is dflash_draft_block's draft. */
dflash_status dflash_draft_block_ids(const dflash_config* cfg, const dflash_weights* w,
                                     const int32_t* ids, const int32_t* ctx_len, int B,
                                     int max_ctx_hint, void* k_cache, void* v_cache, int32_t* draft,
                                     float* logits_opt, int32_t* dev_status, void* ws,
                                     size_t ws_bytes, dflash_trace* trace, dflash_stream_t stream);
dflash_status dflash_unmask_step(const dflash_config* cfg, const float* logits,
                                 const int32_t* draft, int32_t* ids, int B, int steps_left,
                                 void* ws, size_t ws_bytes, dflash_trace* trace,
                                 dflash_stream_t stream);
dflash_status dflash_draft_block_iter(const dflash_config* cfg, const dflash_weights* w,
                                      const int32_t* anchor, const int32_t* ctx_len, int B,
                                      int max_ctx_hint, void* k_cache, void* v_cache, int n_steps,
                                      int32_t* ids, int32_t* draft, float* logits,
                                      int32_t* dev_status, void* ws, size_t ws_bytes,
                                      dflash_trace* trace, dflash_stream_t stream);

/* Sampling mode of the drafting pass (temperature > 0): the pass of
 * dflash_draft_block, except that draft token j of sequence b is a draw from
 * softmax(logits_j / temperature) (the temperature-1 setting of [P1] result
 * tables and [P2]'s lossless rejection-acceptance paragraph), by the
 * Gumbel-max rule: draft = argmax_v (logit_v / T + G_v), G_v = -ln(-ln u_v),
 * u_v = ((z >> 41) + 1/2) 2^-23 with z the splitmix64 output (Steele, Lea,
 * Flood 2014; Vigna's splitmix64.c) of state `seed` at counter
 *   0 << 60 | j << 52 | b << 32 | v          (stream 0: draft sample).
 * logits: device fp32 [B, gamma, V], required: the raw logits (not divided by
 *   T), which dflash_verify_sample needs as the drafter distribution q.
 * Other arguments as in dflash_draft_block (no layer dump). Returns
 * DFLASH_ERR_INVALID_ARG for temperature <= 0 or not finite, or logits NULL. */
dflash_status dflash_draft_block_sample(const dflash_config* cfg, const dflash_weights* w,
                                        const int32_t* anchor, const int32_t* ctx_len, int B,
                                        int max_ctx_hint, void* k_cache, void* v_cache,
                                        float temperature, uint64_t seed, int32_t* draft,
                                        float* logits, int32_t* dev_status, void* ws,
                                        size_t ws_bytes, dflash_trace* trace,
                                        dflash_stream_t stream);

/* Sampling verification (temperature > 0) by rejection-acceptance, which
 * keeps the committed tokens distributed as the target's own sampling
 * ([P2] lossless paragraph; reading: standard speculative sampling):
 *   p_j = softmax(target_logits[b, j] / T),  q_j = softmax(draft_logits[b, j] / T)
 *   for j = 0..gamma-1: keep draft j while u_j q_j(x_j) < p_j(x_j), u_j the
 *     uniform of stream 3 at counter 3 << 60 | j << 52 | b << 32 | 0;
 *   a = kept drafts; tau[b] = a + 1;
 *   a < gamma: y = argmax_v (ln max(p_a(v) - q_a(v), 0) + G_v), stream 1 at
 *     (j = a, v) (entries with no residual mass excluded; if none has mass,
 *     y = argmax_v (target_logits[b, a, v] / T + G_v), same noise);
 *   a = gamma: y = argmax_v (target_logits[b, gamma, v] / T + G_v), stream 2
 *     at (j = gamma, v);
 *   committed[b] = draft[b, 0..a-1] ++ [y] ++ (-1 padding); next_anchor[b] = y.
 * Same generator and uniform as dflash_draft_block_sample. Ties of a draw go
 * to the lowest index. A draft id outside [0, V) counts as rejected.
 * target_logits: device [B, gamma+1, V] of logits_dtype;
 * draft_logits: device fp32 [B, gamma, V] (dflash_draft_block_sample's logits);
 * draft: device [B, gamma]; tau, next_anchor: device [B]; committed: device
 * [B, gamma+1]. Three launches; the workspace holds their scratch. */
dflash_status dflash_verify_sample(const dflash_config* cfg, const void* target_logits,
                                   dflash_dtype logits_dtype, const float* draft_logits,
                                   const int32_t* draft, int B, float temperature,
                                   uint64_t seed, int32_t* tau, int32_t* committed,
                                   int32_t* next_anchor, void* ws, size_t ws_bytes,
                                   dflash_trace* trace, dflash_stream_t stream);

/* Greedy verification, [P1] "Preliminaries" eq. (1) (tau in [1, gamma+1],
 * bonus token included) and "추론 구조" (the target verifies the block):
 *   t_j = argmax_V target_logits[b, j]   (j = 0..gamma; lowest index on ties)
 *   a   = largest k with draft[b, j] == t_j for all j < k
 *   tau[b] = a + 1;  committed[b] = draft[b, 0..a-1] ++ [t_a] ++ (-1 padding)
 *   next_anchor[b] = t_a
 * target_logits: device [B, gamma+1, V] of logits_dtype. Row j is the
 *   target's prediction after the anchor and the first j draft tokens.
 * draft: device [B, gamma]; tau, next_anchor: device [B];
 * committed: device [B, gamma+1]. */
dflash_status dflash_verify_accept(const dflash_config* cfg,
                                   const void* target_logits,
                                   dflash_dtype logits_dtype,
                                   const int32_t* draft, int B, int32_t* tau,
                                   int32_t* committed, int32_t* next_anchor,
                                   void* ws, size_t ws_bytes,
                                   dflash_trace* trace, dflash_stream_t stream);

/* Host helper: fp32 RoPE tables for positions 0..n_pos-1, computed in
 * double precision: cos/sin of p * theta^(-2j/Dh), j = 0..Dh/2-1, row-major
 * [n_pos, Dh/2]. Host pointers; no GPU work. */
dflash_status dflash_rope_tables(const dflash_config* cfg, int n_pos,
                                 float* host_cos, float* host_sin);

/* Plain projection y = x W^T, the building block of every projection above
 * (W_c of [P1] "KV Injection 메커니즘", W^Q/K/V/O and the FFN of the drafter
 * layers). x: [M, K], w: [N, K] of `dtype`; y: [M, N] fp32. K must be a
 * multiple of 64 (bf16) or 32 (fp32). Runs on the same tcgen05 kernel as the
 * drafting step; `ws` needs dflash_workspace_bytes of any valid config. */
dflash_status dflash_linear(dflash_dtype dtype, const void* x, const void* w, float* y, int M,
                            int N, int K, void* ws, size_t ws_bytes, dflash_stream_t stream);

/* Context attention of one drafter layer on its own: the attention step of
 * dflash_draft_block ([P1] "KV Injection 메커니즘", [P4] §3.2), exposed as a
 * building block like dflash_linear (tests, timing of the split-KV kernels):
 *   out[b*R + i, h] = softmax(q[b*R + i, h] . K^T / sqrt(Dh)) V
 * over keys 0 .. ctx_len[b] + gamma of layer `layer`, sequence b and KV head
 * h / (Hq/Hkv) -- the injected context followed by the block's own R rows,
 * which must already be in cache rows ctx_len[b] .. ctx_len[b] + gamma
 * (where dflash_draft_block writes them). No mask, no RoPE (q and the cached
 * K are used as given).
 * q, out: device [B*R, Hq*Dh] of cfg.dtype; ctx_len: device [B];
 * k_cache, v_cache: [L, max_batch, Hkv, Ncap, Dh]; max_ctx_hint as in
 * dflash_draft_block; 0 <= layer < L. The workspace holds the split partials
 * of long contexts. */
dflash_status dflash_attention(const dflash_config* cfg, const void* q, const int32_t* ctx_len, int B,
                               int max_ctx_hint, int layer, const void* k_cache, const void* v_cache,
                               void* out, int32_t* dev_status, void* ws, size_t ws_bytes,
                               dflash_trace* trace, dflash_stream_t stream);

/* Greedy verification without a workspace, for callers that cannot allocate
 * device memory: a serving engine whose memory pool already owns the GPU's
 * memory, a plugin running inside another runtime's step, or a hot loop in
 * which cudaMalloc's implicit device synchronisation is not acceptable. The
 * pages have no counterpart; the computation is that of dflash_verify_accept
 * and the results are identical.
 * Scratch: a fixed array in the library's device memory (about 140 KB per GPU
 * that loads the library, held until the process exits) instead of `ws`.
 * Limits: B <= 1024 and B * (gamma + 1) <= 16384, else DFLASH_ERR_TOO_LARGE
 * and nothing is launched; B <= cfg.max_batch as for dflash_verify_accept
 * (else DFLASH_ERR_INVALID_ARG).
 * Every call looks up the array's address in the current context
 * (cudaGetSymbolAddress, a host-side lookup); the first call in a context
 * loads the library's device code there, so make it before any stream
 * capture. Each call clears the part of the array it uses
 * (cudaMemsetAsync on `stream`) and allocates nothing. All calls share the
 * one array, which keeps the last call's contents: calls whose work overlaps
 * on the GPU (different streams, or concurrent graphs) race on it and must be
 * serialised by the caller. */
dflash_status dflash_verify_accept_noalloc(const dflash_config* cfg,
                                           const void* target_logits,
                                           dflash_dtype logits_dtype,
                                           const int32_t* draft, int B, int32_t* tau,
                                           int32_t* committed, int32_t* next_anchor,
                                           dflash_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H */
