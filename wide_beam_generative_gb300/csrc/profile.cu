// Per-kernel CUDA-event timing for benchmarks (disabled by default).
//
// When enabled, every launcher records an event pair around its kernel on the
// launch stream; beamdec_profile_read sums the elapsed times per kernel.
// Event records are stream-ordered markers and do not change the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace bd {
namespace {

constexpr int kMaxPairs = 8192;
std::mutex g_mu;
bool g_on = false;
unsigned g_mask = 0;   // kernel ids (bits) that get bracketed
int g_n = 0;
cudaEvent_t g_ev[kMaxPairs][2];
int g_kid[kMaxPairs];
bool g_created = false;
int g_open[kKCount];

const char* kNames[kKCount] = {"bd_expand_kernel", "bd_global_kernel", "bd_attn_shared_simt_kernel",
                               "bd_attn_shared_tc_kernel", "bd_attn_merge_kernel",
                               "bd_kv_e4m3_to_bf16_kernel", "bd_stream_select_kernel",
                               "bd_lmhead_kernel", "bd_lmhead_lse_kernel", "bd_seed_kernel"};

}  // namespace

void prof_begin(int kid, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || !((g_mask >> kid) & 1u) || g_n >= kMaxPairs) { g_open[kid] = -1; return; }
  g_kid[g_n] = kid;
  g_open[kid] = g_n;
  cudaEventRecord(g_ev[g_n][0], s);
  ++g_n;
}

void prof_end(int kid, cudaStream_t s) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_on || g_open[kid] < 0) return;
  cudaEventRecord(g_ev[g_open[kid]][1], s);
  g_open[kid] = -1;
}

}  // namespace bd

using namespace bd;

extern "C" int beamdec_profile_enable_mask(unsigned kernel_mask) {
  std::lock_guard<std::mutex> lk(g_mu);
  const bool on = kernel_mask != 0;
  if (on && !g_created) {
    for (int i = 0; i < kMaxPairs; ++i)
      for (int k = 0; k < 2; ++k)
        if (cudaEventCreate(&g_ev[i][k]) != cudaSuccess) return BEAMDEC_ERR_CUDA;
    g_created = true;
  }
  if (on) {   // a new recording starts empty; disabling keeps it for reading
    g_n = 0;
    for (int k = 0; k < kKCount; ++k) g_open[k] = -1;
  }
  g_on = on;
  if (on) g_mask = kernel_mask;
  return BEAMDEC_OK;
}

extern "C" int beamdec_profile_enable(int on) {
  return beamdec_profile_enable_mask(on ? (1u << kKCount) - 1u : 0u);
}

extern "C" int beamdec_profile_read(int kernel_id, float* total_ms, int* launches) {
  if (kernel_id < 0 || kernel_id >= kKCount || total_ms == nullptr || launches == nullptr)
    return BEAMDEC_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  float tot = 0.f;
  int n = 0;
  for (int i = 0; i < g_n; ++i) {
    if (g_kid[i] != kernel_id) continue;
    if (cudaEventSynchronize(g_ev[i][1]) != cudaSuccess) return BEAMDEC_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_ev[i][0], g_ev[i][1]) != cudaSuccess) return BEAMDEC_ERR_CUDA;
    tot += ms;
    ++n;
  }
  *total_ms = tot;
  *launches = n;
  return BEAMDEC_OK;
}

extern "C" const char* beamdec_kernel_name(int kernel_id) {
  if (kernel_id < 0 || kernel_id >= kKCount) return "";
  return kNames[kernel_id];
}
