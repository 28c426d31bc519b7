// beam_select_static: beam_select for callers that cannot allocate device
// memory.  (The pages describe no such variant; it exists for callers of
// this library.)
//
// Some callers only ever see the buffers they are handed: a plugin interface
// of a serving runtime that passes inputs and outputs but no workspace, or a
// process whose device memory is reserved up front by another allocator so
// that cudaMalloc is unavailable or forbidden on the calling path.  For them
// the selection scratch lives in one file-scope device array of fixed size
// (kStaticScratchBytes), which every GPU that loads the library holds until
// the process exits.  Nothing here allocates: no cudaMalloc, no cudaFree, no
// allocating library routine.
//
// The host cannot pass the array's name to a kernel (in host code it is only
// a stand-in symbol, not a device address), so the first call on each device
// resolves the array's device address with cudaGetSymbolAddress while that
// device is current, and caches it with the context it belongs to (a call
// under another context looks the address up again); that first call must
// therefore happen before any stream capture.  After cudaDeviceReset the
// cached address is stale even if the new context reuses the old handle:
// resetting a device under a live process is not supported.
//
// Every call on a device shares the one array and leaves its contents
// behind: each call checks all its arguments first, then clears the 256-byte
// header (status word, barrier counters) on its stream before launching, and
// the selection kernels clear their own counters, so calls that follow one
// another on a stream are independent, while calls that overlap on the GPU
// (different streams, no ordering) race on the array and give undefined
// results.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kStaticScratchBytes = BEAMDEC_STATIC_SELECT_BYTES;   // per device

static __device__ __align__(256) unsigned char g_select_scratch[kStaticScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The context current on the calling thread (null if it cannot be queried):
// the cached address below is only valid inside the context it was resolved in.
CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};
CUcontext g_scratch_ctx[64] = {nullptr};

// Device address of the scratch array in the current device's context,
// looked up with cudaGetSymbolAddress on the first call per device (or when
// the current context is no longer the one the address was taken in).
void* scratch_for_current_device(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *status = BEAMDEC_ERR_CUDA;
    return nullptr;
  }
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || p == nullptr) {
      *status = BEAMDEC_ERR_CUDA;
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = current_context();   // the runtime call above may have made it current
  }
  *status = BEAMDEC_OK;
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" int beam_select_static(const float* logits, int64_t row_stride, const float* lse_in,
                                  const float* cum_in, const int32_t* node_in,
                                  const int32_t* n_live_in, const int32_t* slot_in,
                                  const beamdec_trie* trie, int level, int step, int R, int W,
                                  int K, int V, int T, int32_t* tokens, int32_t* parents,
                                  float* cum_out, float* lse_out, int32_t* node_out,
                                  int32_t* n_live_out, int32_t* slot_out, void* stream) {
  size_t need = 0;
  const int q = beam_select_workspace_size(R, W, K, V, &need);
  if (q != BEAMDEC_OK) return q;
  if (need > kStaticScratchBytes) return BEAMDEC_ERR_UNSUPPORTED;   // larger than the static array
  int status = BEAMDEC_OK;
  void* ws = scratch_for_current_device(&status);
  if (ws == nullptr) return status;
  // every argument is checked before the shared array is touched: a call
  // that is refused writes nothing
  const bd::SelectCall c{logits, row_stride, lse_in, nullptr, cum_in, node_in, n_live_in, slot_in,
                         trie, level, step, R, W, K, V, T, tokens, parents, cum_out, lse_out,
                         node_out, n_live_out, slot_out, ws, kStaticScratchBytes, 0.f, 0};
  bd::SelectArgs a;
  const int rc = bd::select_validate(c, &a);
  if (rc != BEAMDEC_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, bd::kWsHeaderBytesHost, st) != cudaSuccess) return BEAMDEC_ERR_CUDA;
  return bd::launch_select(a, st);
}
