// kda_prefill_static.cu -- kda_prefill with a built-in, statically allocated
// workspace, for callers that cannot allocate device memory themselves.
//
// Who needs it: a host that has already handed every byte of device memory to
// its own pool at start-up (a serving engine reserving its state and cache
// pools), code that issues calls while a CUDA graph is being captured (where
// cudaMalloc is not allowed), and plugin-style callers that receive tensors
// through this C ABI but have no allocator of their own.  This entry point
// allocates nothing: its scratch is the file-scope array below, which every
// GPU that loads the library holds until the process exits.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/kda.h"

namespace {

constexpr size_t kStaticScratchBytes = KDA_PREFILL_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_prefill_scratch[kStaticScratchBytes];

// Device address of g_prefill_scratch on each device, looked up on the first
// call made with that device current.  In host code the array's name is only
// a host-side stand-in, so its device address must come from the runtime.
// Host threads making their first calls at once may each look it up; they
// store the same address, and the atomics keep that well defined.
std::atomic<void*> g_scratch_ptr[kMaxDevices] = {};

kda_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  void* p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
    g_scratch_ptr[dev].store(p, std::memory_order_relaxed);
  }
  *out = p;
  return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_prefill_noalloc(kda_dims dims, kda_gate gate, const kda_bf16* q,
                                          const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                                          const kda_bf16* beta, int64_t gb_rows, float* state_pool,
                                          int pool_slots, const int32_t* state_idx,
                                          const int32_t* cu_seqlens, int num_seqs,
                                          int64_t total_tokens, kda_bf16* o, float* intermediate,
                                          int64_t intermediate_chunks, int32_t* err_flag,
                                          void* stream) {
  // Reject work that does not fit the static scratch before touching anything.
  if (kda_prefill_workspace_size(dims, num_seqs, total_tokens) > kStaticScratchBytes)
    return KDA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const kda_status s = scratch_for_current_device(&scratch);
  if (s != KDA_OK) return s;
  // The prefill clears the flags it uses and writes every other workspace
  // byte it reads within the same call, so nothing left in the array by an
  // earlier call needs clearing here.
  return kda_prefill(dims, gate, q, k, v, g, beta, gb_rows, state_pool, pool_slots, state_idx,
                     cu_seqlens, num_seqs, total_tokens, o, intermediate, intermediate_chunks,
                     scratch, kStaticScratchBytes, err_flag, stream);
}
