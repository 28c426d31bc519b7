// Internal declarations shared by the translation units of libbeamdec.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/beamdec.h"

struct beamdec_trie {
  int levels;
  int32_t vocab;
  int64_t n_items;                        // distinct items
  int32_t C[BEAMDEC_MAX_LEVELS];          // codes per level
  int32_t token_base[BEAMDEC_MAX_LEVELS];
  int64_t n_nodes[BEAMDEC_MAX_LEVELS];    // nodes at level t
  int64_t n_edges[BEAMDEC_MAX_LEVELS];    // edges out of level t = nodes at t+1
  int32_t max_children[BEAMDEC_MAX_LEVELS];
  int32_t* off[BEAMDEC_MAX_LEVELS];       // device [n_nodes+1]
  int32_t* code[BEAMDEC_MAX_LEVELS];      // device [n_edges]
  uint32_t* mask[BEAMDEC_MAX_LEVELS];     // device [n_nodes][mask_words] or null
  int32_t mask_words[BEAMDEC_MAX_LEVELS];
  int device;
};

namespace bd {

// Per-device one-time host set-up (kernel attributes, occupancy queries),
// safe when several host threads make their first call at once: fn(dev)
// runs under a lock until it succeeds once for the current device.
struct PerDeviceOnce {
  std::mutex mu;
  std::atomic<int> done[64] = {};
};
template <class F>
int once_per_device(PerDeviceOnce& o, F&& fn) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BEAMDEC_ERR_CUDA;
  if (o.done[dev].load(std::memory_order_acquire)) return BEAMDEC_OK;
  std::lock_guard<std::mutex> lk(o.mu);
  if (o.done[dev].load(std::memory_order_relaxed)) return BEAMDEC_OK;
  const int rc = fn(dev);
  if (rc == BEAMDEC_OK) o.done[dev].store(1, std::memory_order_release);
  return rc;
}

constexpr size_t kWsHeaderBytesHost = 256;   // status word + grid-barrier counters

// Device view of one trie level for kernels.
struct TrieLevel {
  const int32_t* off;
  const int32_t* code;
  int32_t n_nodes;
  int32_t token_base;
  const uint32_t* mask;   // dense child masks [n_nodes][words], or null (CSR only)
  int32_t words;          // 32-bit words per mask
};

// ---- select ----------------------------------------------------------------
constexpr int kSelectCap = 8192;        // candidate keys sorted by one block
size_t select_workspace_bytes(int R, int W, int K, int V);

struct SelectArgs {
  const float* logits; int64_t row_stride; const float* lse_in;
  // one-launch path only: the normaliser the candidate scores use, given by
  // the caller, while the kernel still streams every row for lse_out
  // (null: the kernel's own log-sum-exp scores the candidates)
  const float* score_lse;
  const float* cum_in; const int32_t* node_in; const int32_t* n_live_in;
  const int32_t* slot_in;
  bool has_trie; TrieLevel lvl;
  int level, step, R, W, K, V, T, Kp;
  int row_splits, row_chunk;   // blocks per logits row and logits per block
  int32_t* tokens; int32_t* parents; float* cum_out; float* lse_out;
  int32_t* node_out; int32_t* n_live_out; int32_t* slot_out;
  void* ws;
  float inv_tau;                  // fl32(1 / temperature); 0 = deterministic top-k
  uint32_t seed_lo, seed_hi;      // Gumbel noise key (temperature > 0)
  // one-launch kernel only: store each live row's scoring normaliser in the
  // workspace and stop (the expansion kernel then selects the rows)
  int lse_only;
  // expansion kernel only: the workspace's seed histogram holds this call's
  // seed of every request's cut (open-vocabulary rows)
  int seeded;
};
int launch_select(const SelectArgs& a, cudaStream_t stream);

// The arguments of one selection call as the C ABI receives them.
struct SelectCall {
  const float* logits; int64_t row_stride; const float* lse_in; const float* score_lse;
  const float* cum_in; const int32_t* node_in; const int32_t* n_live_in; const int32_t* slot_in;
  const beamdec_trie* trie; int level, step, R, W, K, V, T;
  int32_t* tokens; int32_t* parents; float* cum_out; float* lse_out; int32_t* node_out;
  int32_t* n_live_out; int32_t* slot_out;
  void* ws; size_t ws_bytes;
  float temperature;   // 0 = deterministic top-k
  uint64_t seed;
};
// Host-side checks of a selection call (nothing is launched or written);
// on BEAMDEC_OK `a` holds the kernel arguments for launch_select.
int select_validate(const SelectCall& c, SelectArgs* a);

// ---- attention ---------------------------------------------------------------
struct AttnArgs {
  const void* q; const void* shared_k; const void* shared_v;
  const int32_t* prompt_offsets; int max_prompt_len; int64_t shared_rows;
  const void* unshared_k; const void* unshared_v;
  const int32_t* slot_table; const int32_t* n_live;
  int step, R, W, Hq, Hkv, d, T;
  int q_dtype, kv_dtype, out_dtype;
  const float* k_scale; const float* v_scale; float sm_scale;
  void* out; void* ws;
  // e4m3 KV whose prompt part the workspace already holds as bf16
  // (beam_attn_prepare_prompt): the shared stage reads it, no copy is made
  bool kv_prepared;
};
// Split plan of the shared stage over the prompt.
struct AttnPlan {
  int n_split;      // prompt splits (partials per query row)
  int split_len;    // keys per split (multiple of 128)
  bool tensor_core; // tcgen05 shared stage
  bool convert_kv;  // fp8 prompt KV dequantised to bf16 in the workspace first
  int max_prompt_len;
};
AttnPlan attn_plan(int R, int W, int Hq, int Hkv, int d, int max_prompt_len, int q_dtype,
                   int kv_dtype);
size_t attn_workspace_bytes(int R, int W, int Hq, int Hkv, int d, const AttnPlan& p);
int launch_attn_shared_simt(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream);
int launch_attn_shared_tc(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream);
// The bf16 copy of e4m3 prompt K/V in the workspace (and its record of
// shared_k, shared_v, shared_rows and where the copy lies), launched as a
// programmatic dependent; early: the kernel after it may start before it ends.
int launch_kv_copy(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream, bool early);
bool attn_tc_supported(int q_dtype, int kv_dtype, int d, int G);
bool attn_tc_fused(const AttnArgs& a, const AttnPlan& p);   // merge inside the shared stage

// ---- LM head (lmhead.cu) ------------------------------------------------------
size_t lmhead_workspace_bytes(int rows, int V);
int launch_lmhead(const void* hidden, const void* weight, int rows, int hidden_dim, int V,
                  int win0, int win1, float* lse_out, float* logits_out, int64_t out_stride,
                  void* ws, cudaStream_t stream);

// 128-byte-swizzled tiled TMA tensor map (tmap.cu); false if encoding fails.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
              const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box);
int launch_attn_merge(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream);

// Partial-triple layout in the attention workspace (after the 256-byte header):
//   m, l : [n_split][R][Hkv][W*G] fp32 (m in log2 units of the scaled score)
//   o    : [n_split][R][Hkv][W*G][d] fp32, not normalised by l
struct AttnPartials {
  float* m; float* l; float* o;
};
AttnPartials attn_partials(void* ws, int R, int W, int Hq, int Hkv, int d, int n_split);
// bf16 copies of fp8 prompt K then V (R * max_prompt_len rows each), after the partials.
__nv_bfloat16* attn_kv16(void* ws, int R, int W, int Hq, int Hkv, int d, int n_split);

int sm_count();

// ---- per-kernel event timing (off unless beamdec_profile_enable(1)) ---------
enum KernelId { kKExpand = 0, kKGlobal = 1, kKAttnSimt = 2, kKAttnTc = 3, kKAttnMerge = 4,
                kKKvConvert = 5, kKStream = 6, kKLmhead = 7, kKLmheadLse = 8, kKSeed = 9, kKCount = 10 };
void prof_begin(int kid, cudaStream_t s);
void prof_end(int kid, cudaStream_t s);

}  // namespace bd
