// Verify-accept for callers that cannot allocate device memory.
//
// dflash_verify_accept takes its scratch (per-row argmax keys and per-sequence
// arrival counters) from a caller-provided workspace. Some callers cannot
// call cudaMalloc: a serving engine whose memory pool already owns the GPU's
// memory, a plugin that runs inside another runtime's step, or a hot loop in
// which cudaMalloc's implicit device synchronisation is not acceptable. This
// entry point runs the same kernel with its scratch in a fixed-size array in
// the library's own device memory instead, so the caller passes only inputs
// and outputs.
#include "internal.h"

namespace {

constexpr int kNoAllocMaxRows = 16384;  // B * (gamma + 1) rows of target logits per call
constexpr int kNoAllocMaxSeqs = 1024;   // sequences B per call

struct VerifyScratch {
  unsigned long long keys[kNoAllocMaxRows];  // packed (logit, index) argmax per row
  int counters[kNoAllocMaxSeqs];             // CTAs finished per sequence
};

// One copy per GPU that loads the library, held until the process exits
// (about 140 KB). In host code this name is a host-side stand-in, not a
// device address: only the address from cudaGetSymbolAddress is passed on.
static __device__ __align__(256) VerifyScratch g_verify_scratch;

}  // namespace

extern "C" dflash_status dflash_verify_accept_noalloc(const dflash_config* c,
                                                      const void* target_logits,
                                                      dflash_dtype logits_dtype,
                                                      const int32_t* draft, int B, int32_t* tau,
                                                      int32_t* committed, int32_t* next_anchor,
                                                      dflash_stream_t stream) {
  dflash_status st = dflash_check_config(c);
  if (st != DFLASH_OK) return st;
  if (logits_dtype != DFLASH_BF16 && logits_dtype != DFLASH_F32) return DFLASH_ERR_DTYPE;
  if (B < 1 || target_logits == nullptr || draft == nullptr || tau == nullptr ||
      committed == nullptr || next_anchor == nullptr)
    return DFLASH_ERR_INVALID_ARG;
  const int R = c->gamma + 1;
  if (B > kNoAllocMaxSeqs || static_cast<long long>(B) * R > kNoAllocMaxRows)
    return DFLASH_ERR_TOO_LARGE;
  if (B > c->max_batch) return DFLASH_ERR_INVALID_ARG;  // as dflash_verify_accept
  if ((st = dfl::check_arch()) != DFLASH_OK) return st;
  // The array's address in the current context, looked up on every call (a
  // host-side lookup once the module is loaded): an address kept from an
  // earlier call could belong to another context of the same device, or to
  // a context that cudaDeviceReset has since destroyed. The first call in a
  // context loads the module; make it before any stream capture.
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr)
    return DFLASH_ERR_CUDA;
  VerifyScratch* s = static_cast<VerifyScratch*>(p);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // the keys and counters of this call must start at zero
  if (cudaMemsetAsync(s->keys, 0, sizeof(unsigned long long) * B * R, cs) != cudaSuccess ||
      cudaMemsetAsync(s->counters, 0, sizeof(int) * B, cs) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  const cudaError_t e = dfl::launch_verify(target_logits, logits_dtype == DFLASH_BF16, draft, nullptr, B,
                                           c->gamma, c->vocab, tau, committed, next_anchor, s->keys,
                                           s->counters, cs, dfl::use_pdl());
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}
