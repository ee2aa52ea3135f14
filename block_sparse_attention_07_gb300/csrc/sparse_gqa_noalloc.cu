// msa_sparse_gqa_decode_noalloc: the sparse GQA decode of msa_sparse_gqa_decode
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs where allocation
// is forbidden or unavailable (inside a memory-capped serving process whose
// allocator owns every byte, in a plugin that gets only input/output buffers
// from its host framework, or in tooling that must not change the device's
// memory footprint during a run). This entry point serves them: it takes the
// same inputs and outputs as msa_sparse_gqa_decode but no workspace. Its
// split-K partials live in a fixed file-scope device array, g_gqa_scratch, of
// kNoAllocScratchBytes (64 MiB). Every GPU that loads the library holds this
// array until the process exits.
//
// Rules that follow from the shared array:
//   - The first call on a device looks up the array's device address with
//     cudaGetSymbolAddress (with that device current) and remembers it; make
//     that first call before any stream capture on that device. The address
//     belongs to the device's current context: when that context changes (a
//     cudaDeviceReset, a new primary context), the next call looks it up again,
//     so that call too should come before any stream capture.
//   - Every call on a device uses the same array. The partials need no
//     initial value (each is written before it is read) and the array keeps the
//     last call's contents, but two calls whose kernels overlap on the GPU (on
//     different streams, or from different threads) race on it: serialise them.
//   - A shape whose workspace does not fit (B * Q * G * (topk * 8,320 + 8)
//     bytes > 64 MiB) is rejected with MSA_ERR_WORKSPACE before anything is
//     launched.
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda.h>

#include <mutex>

#include "msa_internal.h"

namespace msa {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;

static __device__ __align__(256) float g_gqa_scratch[kNoAllocScratchBytes / sizeof(float)];

// Unique id of the calling thread's current context (driver calls looked up
// through the runtime, as the library does not link libcuda). False when the
// driver does not offer them.
static bool current_context_id(unsigned long long* id) {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_gqa_scratch on the current device, looked up once per
// device and context (every call, if the context id is not available).
static cudaError_t scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[128] = {nullptr};
  static unsigned long long ctx_of[128] = {0};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  unsigned long long ctx = 0;
  const bool known = current_context_id(&ctx);   // false too before the runtime has made a context current
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || !known || ctx_of[dev] != ctx) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_gqa_scratch);   // makes the device's primary context current if none is
    if (err != cudaSuccess) return err;
    addr[dev] = p;
    ctx_of[dev] = current_context_id(&ctx) ? ctx : 0;
  }
  *out = addr[dev];
  return cudaSuccess;
}

}  // namespace msa

using namespace msa;

extern "C" msa_status_t msa_sparse_gqa_decode_noalloc(const msa_dims_t* dims, const void* q,
                                                      const msa_kv_cache_t* cache, const int32_t* block_table,
                                                      const int32_t* seq_lens, const int32_t* selected, void* out,
                                                      float* lse, uint32_t* dev_flags, void* stream) {
  if (dims == nullptr) return MSA_ERR_INVALID_ARG;
  const size_t need = msa_sparse_gqa_workspace_size(dims, cache != nullptr ? cache->dtype : MSA_BF16);
  if (need == 0) return msa_sparse_gqa_decode(dims, q, cache, block_table, seq_lens, selected, out, lse, nullptr,
                                              0, dev_flags, stream);   // reports the shape error
  if (need > kNoAllocScratchBytes) return MSA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MSA_ERR_CUDA;
  return msa_sparse_gqa_decode(dims, q, cache, block_table, seq_lens, selected, out, lse, scratch,
                               kNoAllocScratchBytes, dev_flags, stream);
}
