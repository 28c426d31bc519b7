// C ABI of libbeamdec: argument validation, workspace sizing and dispatch.
#include <cuda_runtime.h>
#include <math.h>

#include <cuda_bf16.h>

#include "internal.h"

namespace bd {

int sm_count() {
  static std::atomic<int> cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {   // every thread that races here stores the same value
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static size_t a256(size_t x) { return (x + 255) & ~(size_t)255; }

AttnPlan attn_plan(int R, int W, int Hq, int Hkv, int d, int max_prompt_len, int q_dtype,
                   int kv_dtype) {
  // The plan depends on shapes only (never on the device), so the workspace
  // size query and the call always agree.
  AttnPlan p;
  const int G = Hq / Hkv;
  p.tensor_core = attn_tc_supported(q_dtype, kv_dtype, d, G);
  const int rows = W * G;
  const int tile_rows = p.tensor_core ? 256 : 32;
  const long long units = (long long)R * Hkv * ((rows + tile_rows - 1) / tile_rows);
  const long long sms = 152;   // GB300 SM count, a planning constant
  const int chunk = 128;
  const int chunks = max_prompt_len > 0 ? (max_prompt_len + chunk - 1) / chunk : 1;
  // split count from a small time model (microseconds): each wave of CTAs
  // costs its chunks (about 1.75 us per 128 keys for a 256-row tile on the
  // tensor cores, measured in a busy kernel) plus a 2 us prologue; every
  // split's partial triples are read back by the merge at about 6 TB/s, and
  // each split adds about 0.5 us of the merge's dependent reads (a 1 x 50
  // beam, 2048-key step measured 50.0 / 46.0 / 47.8 / 54.3 us at 16 / 8 / 4
  // / 2 splits).
  const double chunk_us = p.tensor_core ? 1.75 : 4.0;
  const double part_us = (double)R * Hkv * rows * (d + 2) * 4 / 6.0e6 + 0.5;
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= 16 && s <= chunks; ++s) {
    const long long waves = (units * s + sms - 1) / sms;
    const long long per = (chunks + s - 1) / s;
    const double cost = (double)waves * (per * chunk_us + 2.0) + s * part_us;
    if (cost < best_cost - 1e-9) { best_cost = cost; best = s; }
  }
  p.split_len = ((chunks + best - 1) / best) * chunk;
  p.convert_kv = p.tensor_core && kv_dtype == BEAMDEC_E4M3;
  p.max_prompt_len = max_prompt_len;
  p.n_split = max_prompt_len > 0 ? (max_prompt_len + p.split_len - 1) / p.split_len : 1;
  (void)d;
  return p;
}

size_t attn_workspace_bytes(int R, int W, int Hq, int Hkv, int d, const AttnPlan& p) {
  const size_t rows = (size_t)R * Hkv * W * (Hq / Hkv) * p.n_split;
  const size_t kv16 = p.convert_kv ? a256((size_t)2 * R * p.max_prompt_len * Hkv * d * 2) : 0;
  return kWsHeaderBytesHost + a256(rows * 4) * 2 + a256(rows * d * 4) + kv16;
}

__nv_bfloat16* attn_kv16(void* ws, int R, int W, int Hq, int Hkv, int d, int n_split) {
  const size_t rows = (size_t)R * Hkv * W * (Hq / Hkv) * n_split;
  char* p = static_cast<char*>(ws) + kWsHeaderBytesHost + a256(rows * 4) * 2 + a256(rows * d * 4);
  return reinterpret_cast<__nv_bfloat16*>(p);
}

AttnPartials attn_partials(void* ws, int R, int W, int Hq, int Hkv, int d, int n_split) {
  const size_t rows = (size_t)R * Hkv * W * (Hq / Hkv) * n_split;
  char* p = static_cast<char*>(ws) + kWsHeaderBytesHost;
  AttnPartials a;
  a.m = reinterpret_cast<float*>(p);
  p += a256(rows * 4);
  a.l = reinterpret_cast<float*>(p);
  p += a256(rows * 4);
  a.o = reinterpret_cast<float*>(p);
  (void)d;
  return a;
}

}  // namespace bd

using namespace bd;

extern "C" const char* beamdec_error_string(int s) {
  switch (s) {
    case BEAMDEC_OK: return "ok";
    case BEAMDEC_ERR_INVALID_ARG: return "invalid argument";
    case BEAMDEC_ERR_UNSUPPORTED: return "unsupported shape or type";
    case BEAMDEC_ERR_WORKSPACE: return "workspace too small";
    case BEAMDEC_ERR_CUDA: return "CUDA runtime error";
    case BEAMDEC_ERR_TIMEOUT: return "bounded device wait timed out";
    case BEAMDEC_ERR_DEVICE_CHECK: return "device-side index check failed";
    case BEAMDEC_ERR_ALLOC: return "device allocation failed";
    default: return "unknown status";
  }
}

extern "C" const char* beamdec_version(void) { return "0.1.0"; }

extern "C" int beamdec_read_status(void* workspace, void* stream_ptr, int32_t* host_status) {
  if (workspace == nullptr || host_status == nullptr) return BEAMDEC_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess ||
      cudaMemsetAsync(workspace, 0, sizeof(v), stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return BEAMDEC_ERR_CUDA;
  *host_status = v;
  return BEAMDEC_OK;
}

extern "C" int beam_select_workspace_size(int R, int W, int K, int V, size_t* bytes) {
  if (bytes == nullptr || R < 1 || W < 1 || K < 1 || V < 1) return BEAMDEC_ERR_INVALID_ARG;
  if (W > BEAMDEC_MAX_BEAM_WIDTH || V > BEAMDEC_MAX_VOCAB) return BEAMDEC_ERR_UNSUPPORTED;
  *bytes = select_workspace_bytes(R, W, K, V);
  return BEAMDEC_OK;
}

namespace bd {

int select_validate(const SelectCall& c, SelectArgs* out) {
  if (c.logits == nullptr || c.cum_in == nullptr || c.n_live_in == nullptr || c.tokens == nullptr ||
      c.parents == nullptr || c.cum_out == nullptr || c.node_out == nullptr ||
      c.n_live_out == nullptr || c.slot_out == nullptr || c.ws == nullptr)
    return BEAMDEC_ERR_INVALID_ARG;
  if (c.R < 1 || c.W < 1 || c.K < 1 || c.V < 1 || c.T < 1 || c.step < 0 || c.step >= c.T ||
      c.row_stride < c.V)
    return BEAMDEC_ERR_INVALID_ARG;
  if (c.step > 0 && c.slot_in == nullptr) return BEAMDEC_ERR_INVALID_ARG;
  if (c.slot_in != nullptr && c.slot_in == c.slot_out) return BEAMDEC_ERR_INVALID_ARG;
  // outputs are written while other blocks still read the inputs
  if (c.cum_out == c.cum_in || (const void*)c.n_live_out == (const void*)c.n_live_in ||
      (c.node_in != nullptr && (const void*)c.node_out == (const void*)c.node_in))
    return BEAMDEC_ERR_INVALID_ARG;
  if (c.lse_in != nullptr && c.score_lse != nullptr) return BEAMDEC_ERR_INVALID_ARG;
  if (c.W > BEAMDEC_MAX_BEAM_WIDTH || c.V > BEAMDEC_MAX_VOCAB) return BEAMDEC_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(c.ws) & 255u) != 0) return BEAMDEC_ERR_INVALID_ARG;
  SelectArgs a{};
  a.has_trie = c.trie != nullptr;
  if (a.has_trie) {
    const beamdec_trie* trie = c.trie;
    if (c.node_in == nullptr || c.level < 0 || c.level >= trie->levels) return BEAMDEC_ERR_INVALID_ARG;
    if (trie->vocab != c.V) return BEAMDEC_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BEAMDEC_ERR_CUDA;
    if (dev != trie->device) return BEAMDEC_ERR_INVALID_ARG;
    a.lvl.off = trie->off[c.level];
    a.lvl.code = trie->code[c.level];
    a.lvl.n_nodes = (int32_t)trie->n_nodes[c.level];
    a.lvl.token_base = trie->token_base[c.level];
    a.lvl.mask = trie->mask[c.level];
    a.lvl.words = trie->mask_words[c.level];
  }
  if (c.ws_bytes < select_workspace_bytes(c.R, c.W, c.K, c.V)) return BEAMDEC_ERR_WORKSPACE;
  a.logits = c.logits; a.row_stride = c.row_stride; a.lse_in = c.lse_in; a.score_lse = c.score_lse;
  a.cum_in = c.cum_in; a.node_in = c.node_in; a.n_live_in = c.n_live_in; a.slot_in = c.slot_in;
  a.level = c.level; a.step = c.step; a.R = c.R; a.W = c.W; a.K = c.K; a.V = c.V; a.T = c.T;
  a.Kp = c.K < c.V ? c.K : c.V;
  a.tokens = c.tokens; a.parents = c.parents; a.cum_out = c.cum_out; a.lse_out = c.lse_out;
  a.node_out = c.node_out; a.n_live_out = c.n_live_out; a.slot_out = c.slot_out;
  a.ws = c.ws;
  a.inv_tau = c.temperature > 0.f ? (float)(1.0 / (double)c.temperature) : 0.f;
  a.seed_lo = (uint32_t)(c.seed & 0xFFFFFFFFull);
  a.seed_hi = (uint32_t)(c.seed >> 32);
  *out = a;
  return BEAMDEC_OK;
}

}  // namespace bd

static int check_temperature(float temperature) {
  if (!(temperature > 0.f) || !(temperature < INFINITY)) return BEAMDEC_ERR_INVALID_ARG;
  if (!((float)(1.0 / (double)temperature) < INFINITY)) return BEAMDEC_ERR_INVALID_ARG;
  return BEAMDEC_OK;
}

static int select_run(const SelectCall& c, void* stream) {
  SelectArgs a;
  const int rc = select_validate(c, &a);
  if (rc != BEAMDEC_OK) return rc;
  return launch_select(a, static_cast<cudaStream_t>(stream));
}

extern "C" int beam_select(const float* logits, int64_t row_stride, const float* lse_in,
                           const float* cum_in, const int32_t* node_in,
                           const int32_t* n_live_in, const int32_t* slot_in,
                           const beamdec_trie* trie, int level, int step, int R, int W, int K,
                           int V, int T, int32_t* tokens, int32_t* parents, float* cum_out,
                           float* lse_out, int32_t* node_out, int32_t* n_live_out,
                           int32_t* slot_out, void* workspace, size_t workspace_bytes,
                           void* stream) {
  const SelectCall c{logits, row_stride, lse_in, nullptr, cum_in, node_in, n_live_in, slot_in,
                     trie, level, step, R, W, K, V, T, tokens, parents, cum_out, lse_out,
                     node_out, n_live_out, slot_out, workspace, workspace_bytes, 0.f, 0};
  return select_run(c, stream);
}

extern "C" int beam_select_gumbel(const float* logits, int64_t row_stride, const float* lse_in,
                                  const float* cum_in, const int32_t* node_in,
                                  const int32_t* n_live_in, const int32_t* slot_in,
                                  const beamdec_trie* trie, int level, int step, int R, int W,
                                  int K, int V, int T, float temperature, uint64_t seed,
                                  int32_t* tokens, int32_t* parents, float* cum_out,
                                  float* lse_out, int32_t* node_out, int32_t* n_live_out,
                                  int32_t* slot_out, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  const int tc = check_temperature(temperature);
  if (tc != BEAMDEC_OK) return tc;
  const SelectCall c{logits, row_stride, lse_in, nullptr, cum_in, node_in, n_live_in, slot_in,
                     trie, level, step, R, W, K, V, T, tokens, parents, cum_out, lse_out,
                     node_out, n_live_out, slot_out, workspace, workspace_bytes, temperature, seed};
  return select_run(c, stream);
}

extern "C" int beam_select_fixed_lse(const float* logits, int64_t row_stride, const float* score_lse,
                                     const float* cum_in, const int32_t* node_in,
                                     const int32_t* n_live_in, const int32_t* slot_in,
                                     const beamdec_trie* trie, int level, int step, int R, int W,
                                     int K, int V, int T, float temperature, uint64_t seed,
                                     int32_t* tokens, int32_t* parents, float* cum_out,
                                     float* lse_out, int32_t* node_out, int32_t* n_live_out,
                                     int32_t* slot_out, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  if (score_lse == nullptr) return BEAMDEC_ERR_INVALID_ARG;
  if (temperature != 0.f) {
    const int tc = check_temperature(temperature);
    if (tc != BEAMDEC_OK) return tc;
  }
  const SelectCall c{logits, row_stride, nullptr, score_lse, cum_in, node_in, n_live_in, slot_in,
                     trie, level, step, R, W, K, V, T, tokens, parents, cum_out, lse_out,
                     node_out, n_live_out, slot_out, workspace, workspace_bytes, temperature, seed};
  return select_run(c, stream);
}

static bool attn_types_ok(int q, int kv, int o) {
  return (q == BEAMDEC_F32 && kv == BEAMDEC_F32 && o == BEAMDEC_F32) ||
         (q == BEAMDEC_BF16 && kv == BEAMDEC_BF16 && o == BEAMDEC_BF16) ||
         (q == BEAMDEC_BF16 && kv == BEAMDEC_E4M3 && o == BEAMDEC_BF16);
}

static int attn_shape_check(int R, int W, int Hq, int Hkv, int d, int max_prompt_len) {
  if (R < 1 || W < 1 || Hq < 1 || Hkv < 1 || d < 1 || max_prompt_len < 0)
    return BEAMDEC_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return BEAMDEC_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || Hq / Hkv > 16 || W > BEAMDEC_MAX_BEAM_WIDTH)
    return BEAMDEC_ERR_UNSUPPORTED;
  return BEAMDEC_OK;
}

extern "C" int beam_attn_workspace_size(int R, int W, int Hq, int Hkv, int d, int max_prompt_len,
                                        int kv_dtype, size_t* bytes) {
  if (bytes == nullptr) return BEAMDEC_ERR_INVALID_ARG;
  const int s = attn_shape_check(R, W, Hq, Hkv, d, max_prompt_len);
  if (s != BEAMDEC_OK) return s;
  if (kv_dtype < BEAMDEC_F32 || kv_dtype > BEAMDEC_E4M3_PREPARED) return BEAMDEC_ERR_INVALID_ARG;
  if (kv_dtype == BEAMDEC_E4M3_PREPARED) kv_dtype = BEAMDEC_E4M3;   // the same layout
  const int q_dtype = kv_dtype == BEAMDEC_F32 ? BEAMDEC_F32 : BEAMDEC_BF16;
  AttnPlan p = attn_plan(R, W, Hq, Hkv, d, max_prompt_len, q_dtype, kv_dtype);
  *bytes = attn_workspace_bytes(R, W, Hq, Hkv, d, p);
  return BEAMDEC_OK;
}

extern "C" int beam_attn_decode(const void* q, const void* shared_k, const void* shared_v,
                                const int32_t* prompt_offsets, int max_prompt_len,
                                int64_t shared_rows, const void* unshared_k, const void* unshared_v,
                                const int32_t* slot_table, const int32_t* n_live, int step,
                                int R, int W, int Hq, int Hkv, int d, int T, int q_dtype,
                                int kv_dtype, int out_dtype, const float* k_scale,
                                const float* v_scale, float sm_scale, void* out,
                                void* workspace, size_t workspace_bytes, void* stream) {
  if (q == nullptr || prompt_offsets == nullptr || unshared_k == nullptr ||
      unshared_v == nullptr || slot_table == nullptr || n_live == nullptr || out == nullptr ||
      workspace == nullptr)
    return BEAMDEC_ERR_INVALID_ARG;
  if (max_prompt_len > 0 && (shared_k == nullptr || shared_v == nullptr))
    return BEAMDEC_ERR_INVALID_ARG;
  if (shared_rows < 0 || (max_prompt_len > 0 && shared_rows < max_prompt_len) ||
      shared_rows > (int64_t)R * max_prompt_len)
    return BEAMDEC_ERR_INVALID_ARG;
  const int s = attn_shape_check(R, W, Hq, Hkv, d, max_prompt_len);
  if (s != BEAMDEC_OK) return s;
  if (T < 1 || step < 0 || step >= T) return BEAMDEC_ERR_INVALID_ARG;
  // the prepared form of e4m3 KV: its prompt part is already in the
  // workspace as bf16 (beam_attn_prepare_prompt)
  const bool prepared = kv_dtype == BEAMDEC_E4M3_PREPARED;
  if (prepared) kv_dtype = BEAMDEC_E4M3;
  if (!attn_types_ok(q_dtype, kv_dtype, out_dtype)) {
    const bool enums_ok = q_dtype >= 0 && q_dtype <= 2 && kv_dtype >= 0 && kv_dtype <= 2 &&
                          out_dtype >= 0 && out_dtype <= 2;
    return enums_ok ? BEAMDEC_ERR_UNSUPPORTED : BEAMDEC_ERR_INVALID_ARG;
  }
  if (kv_dtype == BEAMDEC_E4M3 && (k_scale == nullptr || v_scale == nullptr))
    return BEAMDEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return BEAMDEC_ERR_INVALID_ARG;
  AttnPlan p = attn_plan(R, W, Hq, Hkv, d, max_prompt_len, q_dtype, kv_dtype);
  if (workspace_bytes < attn_workspace_bytes(R, W, Hq, Hkv, d, p)) return BEAMDEC_ERR_WORKSPACE;
  AttnArgs a{};
  a.q = q; a.shared_k = shared_k; a.shared_v = shared_v;
  a.prompt_offsets = prompt_offsets; a.max_prompt_len = max_prompt_len; a.shared_rows = shared_rows;
  a.unshared_k = unshared_k; a.unshared_v = unshared_v;
  a.slot_table = slot_table; a.n_live = n_live;
  a.step = step; a.R = R; a.W = W; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.T = T;
  a.q_dtype = q_dtype; a.kv_dtype = kv_dtype; a.out_dtype = out_dtype;
  a.k_scale = k_scale; a.v_scale = v_scale;
  a.sm_scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf((float)d);
  a.out = out; a.ws = workspace;
  a.kv_prepared = prepared && p.convert_kv;   // shapes without the bf16 copy read fp8 directly
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = p.tensor_core ? launch_attn_shared_tc(a, p, st) : launch_attn_shared_simt(a, p, st);
  if (rc != BEAMDEC_OK) return rc;
  if (p.tensor_core && attn_tc_fused(a, p)) return BEAMDEC_OK;   // merged in the shared stage
  return launch_attn_merge(a, p, st);
}

extern "C" int beam_attn_prepare_prompt(const void* shared_k, const void* shared_v,
                                        const int32_t* prompt_offsets, int max_prompt_len,
                                        int64_t shared_rows, int R, int W, int Hq, int Hkv, int d,
                                        int kv_dtype, void* workspace, size_t workspace_bytes,
                                        void* stream) {
  if (prompt_offsets == nullptr || workspace == nullptr) return BEAMDEC_ERR_INVALID_ARG;
  const int s = attn_shape_check(R, W, Hq, Hkv, d, max_prompt_len);
  if (s != BEAMDEC_OK) return s;
  if (kv_dtype < BEAMDEC_F32 || kv_dtype > BEAMDEC_E4M3) return BEAMDEC_ERR_INVALID_ARG;
  if (shared_rows < 0 || (max_prompt_len > 0 && shared_rows < max_prompt_len) ||
      shared_rows > (int64_t)R * max_prompt_len)
    return BEAMDEC_ERR_INVALID_ARG;
  if (shared_rows > 0 && (shared_k == nullptr || shared_v == nullptr)) return BEAMDEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return BEAMDEC_ERR_INVALID_ARG;
  if (kv_dtype != BEAMDEC_E4M3) return BEAMDEC_OK;   // nothing to prepare
  AttnPlan p = attn_plan(R, W, Hq, Hkv, d, max_prompt_len, BEAMDEC_BF16, kv_dtype);
  if (workspace_bytes < attn_workspace_bytes(R, W, Hq, Hkv, d, p)) return BEAMDEC_ERR_WORKSPACE;
  if (!p.convert_kv || shared_rows == 0) return BEAMDEC_OK;   // no bf16 copy is read at this shape
  if (((reinterpret_cast<uintptr_t>(shared_k) | reinterpret_cast<uintptr_t>(shared_v)) & 15u) != 0)
    return BEAMDEC_ERR_INVALID_ARG;   // read in 16-byte groups, as beam_attn_decode does
  AttnArgs a{};
  a.shared_k = shared_k; a.shared_v = shared_v; a.prompt_offsets = prompt_offsets;
  a.max_prompt_len = max_prompt_len; a.shared_rows = shared_rows;
  a.R = R; a.W = W; a.Hq = Hq; a.Hkv = Hkv; a.d = d;
  a.q_dtype = BEAMDEC_BF16; a.kv_dtype = kv_dtype; a.out_dtype = BEAMDEC_BF16;
  a.ws = workspace;
  return launch_kv_copy(a, p, static_cast<cudaStream_t>(stream), false);
}

// ---- LM head with fused log-sum-exp ---------------------------------------------

extern "C" int beam_lmhead_workspace_size(int rows, int V, size_t* bytes) {
  if (bytes == nullptr || rows < 1 || V < 1) return BEAMDEC_ERR_INVALID_ARG;
  *bytes = bd::lmhead_workspace_bytes(rows, V);
  return BEAMDEC_OK;
}

extern "C" int beam_lmhead_lse(const void* hidden, const void* weight, int rows, int hidden_dim,
                               int V, int window_start, int window_len, float* lse_out,
                               float* logits_out, int64_t logits_row_stride, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (hidden == nullptr || weight == nullptr || lse_out == nullptr || workspace == nullptr)
    return BEAMDEC_ERR_INVALID_ARG;
  if (rows < 1 || V < 1 || hidden_dim < 64 || window_start < 0 || window_len < 0 ||
      (int64_t)window_start + window_len > V)
    return BEAMDEC_ERR_INVALID_ARG;
  if (hidden_dim % 64 != 0 || V > BEAMDEC_MAX_VOCAB || hidden_dim > 65536) return BEAMDEC_ERR_UNSUPPORTED;
  if (window_len > 0 && (logits_out == nullptr || logits_row_stride < (int64_t)window_start + window_len))
    return BEAMDEC_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(hidden) & 15u) || (reinterpret_cast<uintptr_t>(weight) & 15u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return BEAMDEC_ERR_INVALID_ARG;
  if (workspace_bytes < bd::lmhead_workspace_bytes(rows, V)) return BEAMDEC_ERR_WORKSPACE;
  return bd::launch_lmhead(hidden, weight, rows, hidden_dim, V, window_start,
                           window_start + window_len, lse_out, window_len > 0 ? logits_out : nullptr,
                           logits_row_stride, workspace, static_cast<cudaStream_t>(stream));
}
