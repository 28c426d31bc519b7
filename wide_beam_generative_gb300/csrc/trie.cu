// Catalog trie construction (canonical CSR, one level per decode step).
//
// "Generative recommendation design" (xLLM) §4.3: invalid item paths are
// filtered before they become candidates; FlashRec (SGLang PR 31626 thread):
// a fused SID trie in CSR form keeps the illegal-SID rate at 0.
//
// The catalog is preprocessed once, not per decode step: items are sorted
// lexicographically (packed into 64-bit keys when the code widths fit, and
// then sorted in slices on the host's cores and merged), de-duplicated, and each level's CSR is read off the sorted order: sorted item
// i opens a new length-(t+1) prefix (an edge of level t) exactly when it
// differs from item i-1 within its first t+1 codes.  The CSR arrays are then
// uploaded to device memory owned by the handle.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <new>
#include <numeric>
#include <thread>
#include <utility>
#include <vector>

#include "internal.h"

namespace {

int bits_for(int32_t C) {
  int b = 0;
  while ((1ll << b) < (long long)C) ++b;
  return b;
}

// Ascending sort of (key, index) pairs: slices sorted on up to 16 threads,
// then merged pairwise in rounds; the pairs are distinct (the index breaks
// ties), so the result is the unique ascending order whatever the slicing.
// Falls back to one thread when a thread cannot be started.
void sort_pairs(std::vector<std::pair<uint64_t, int64_t>>& v) {
  const int64_t n = (int64_t)v.size();
  unsigned T = std::thread::hardware_concurrency();
  T = T < 1 ? 1 : (T > 16 ? 16 : T);
  if (n < (1 << 16) || T == 1) {
    std::sort(v.begin(), v.end());
    return;
  }
  std::vector<int64_t> b(T + 1);
  for (unsigned i = 0; i <= T; ++i) b[i] = n * (int64_t)i / (int64_t)T;
  auto run_all = [](std::vector<std::thread>& th) {
    for (auto& t : th) t.join();
  };
  try {
    std::vector<std::thread> th;
    for (unsigned t = 0; t < T; ++t)
      th.emplace_back([&v, &b, t] { std::sort(v.begin() + b[t], v.begin() + b[t + 1]); });
    run_all(th);
    for (unsigned w = 1; w < T; w *= 2) {
      std::vector<std::thread> mt;
      for (unsigned t = 0; t + w < T; t += 2 * w) {
        const int64_t lo = b[t], mid = b[t + w], hi = b[std::min(t + 2 * w, T)];
        mt.emplace_back([&v, lo, mid, hi] { std::inplace_merge(v.begin() + lo, v.begin() + mid, v.begin() + hi); });
      }
      run_all(mt);
    }
  } catch (...) {   // a thread could not be started (the joins above never throw)
    std::sort(v.begin(), v.end());
  }
}

}  // namespace

extern "C" int beam_trie_build(const int32_t* items, int64_t n_items, int levels,
                               const int32_t* codes_per_level, const int32_t* token_base,
                               int32_t vocab, void* stream_ptr, beamdec_trie** out) {
  if (out == nullptr) return BEAMDEC_ERR_INVALID_ARG;
  *out = nullptr;
  if (items == nullptr || codes_per_level == nullptr || token_base == nullptr || n_items < 1 ||
      levels < 1 || vocab < 1)
    return BEAMDEC_ERR_INVALID_ARG;
  if (levels > BEAMDEC_MAX_LEVELS || vocab > BEAMDEC_MAX_VOCAB || n_items >= (1ll << 31))
    return BEAMDEC_ERR_UNSUPPORTED;
  int total_bits = 0;
  for (int l = 0; l < levels; ++l) {
    const int32_t C = codes_per_level[l];
    if (C < 1 || token_base[l] < 0) return BEAMDEC_ERR_INVALID_ARG;
    if (C > BEAMDEC_MAX_CODES) return BEAMDEC_ERR_UNSUPPORTED;
    if ((int64_t)token_base[l] + C > vocab) return BEAMDEC_ERR_INVALID_ARG;
    total_bits += bits_for(C);
  }
  for (int64_t i = 0; i < n_items * levels; ++i) {
    const int l = (int)(i % levels);
    if (items[i] < 0 || items[i] >= codes_per_level[l]) return BEAMDEC_ERR_INVALID_ARG;
  }
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);

  // lexicographic order of the items
  std::vector<int64_t> order(n_items);
  if (total_bits <= 64) {
    std::vector<std::pair<uint64_t, int64_t>> kp(n_items);
    for (int64_t i = 0; i < n_items; ++i) {
      uint64_t k = 0;
      for (int l = 0; l < levels; ++l)
        k = (total_bits ? (k << bits_for(codes_per_level[l])) : 0) | (uint64_t)items[i * levels + l];
      kp[i] = {k, i};
    }
    sort_pairs(kp);
    for (int64_t i = 0; i < n_items; ++i) order[i] = kp[i].second;
  } else {
    std::iota(order.begin(), order.end(), 0);
    std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
      const int32_t* x = items + a * levels;
      const int32_t* y = items + b * levels;
      for (int l = 0; l < levels; ++l)
        if (x[l] != y[l]) return x[l] < y[l];
      return a < b;
    });
  }
  // first differing level of each sorted item against its predecessor
  // (levels = identical, i.e. a duplicate)
  std::vector<int64_t> uniq;
  std::vector<int8_t> diff;
  uniq.reserve(n_items);
  diff.reserve(n_items);
  for (int64_t k = 0; k < n_items; ++k) {
    const int32_t* x = items + order[k] * levels;
    int dl = 0;
    if (k > 0) {
      const int32_t* y = items + order[k - 1] * levels;
      while (dl < levels && x[dl] == y[dl]) ++dl;
      if (dl == levels) continue;   // duplicate
    }
    uniq.push_back(order[k]);
    diff.push_back((int8_t)dl);
  }
  const int64_t n = (int64_t)uniq.size();

  beamdec_trie* t = new (std::nothrow) beamdec_trie();
  if (t == nullptr) return BEAMDEC_ERR_ALLOC;
  std::memset(t, 0, sizeof(*t));
  t->levels = levels;
  t->vocab = vocab;
  t->n_items = n;
  cudaGetDevice(&t->device);
  int status = BEAMDEC_OK;
  std::vector<int32_t> off, code;
  for (int lv = 0; lv < levels && status == BEAMDEC_OK; ++lv) {
    t->C[lv] = codes_per_level[lv];
    t->token_base[lv] = token_base[lv];
    // nodes at level lv = items opening a new lv-prefix (diff < lv); the root for lv = 0
    off.assign(1, 0);
    code.clear();
    int64_t node = -1;
    for (int64_t k = 0; k < n; ++k) {
      const int d = diff[k];
      if (lv == 0 ? k == 0 : d < lv) {   // new node at this level
        ++node;
        off.push_back(off.back());
      }
      if (d <= lv) {                      // new edge (a new (lv+1)-prefix)
        code.push_back(items[uniq[k] * levels + lv]);
        off.back() += 1;
      }
    }
    t->n_nodes[lv] = node + 1;
    t->n_edges[lv] = (int64_t)code.size();
    int32_t mx = 0;
    for (size_t i = 0; i + 1 < off.size(); ++i) mx = std::max(mx, off[i + 1] - off[i]);
    t->max_children[lv] = mx;
    if (cudaMalloc(&t->off[lv], off.size() * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&t->code[lv], code.size() * sizeof(int32_t)) != cudaSuccess) {
      status = BEAMDEC_ERR_ALLOC;
      break;
    }
    if (cudaMemcpyAsync(t->off[lv], off.data(), off.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaMemcpyAsync(t->code[lv], code.data(), code.size() * sizeof(int32_t),
                        cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
      status = BEAMDEC_ERR_CUDA;
      break;
    }
  }
  if (status != BEAMDEC_OK) {
    beam_trie_free(t);
    return status;
  }
  *out = t;
  return BEAMDEC_OK;
}

extern "C" void beam_trie_free(beamdec_trie* t) {
  if (t == nullptr) return;
  for (int l = 0; l < BEAMDEC_MAX_LEVELS; ++l) {
    if (t->off[l]) cudaFree(t->off[l]);
    if (t->code[l]) cudaFree(t->code[l]);
    if (t->mask[l]) cudaFree(t->mask[l]);
  }
  delete t;
}

extern "C" int beam_trie_info(const beamdec_trie* t, int* levels, int32_t* vocab,
                              int64_t* n_distinct, int64_t* n_nodes, int64_t* n_edges,
                              int32_t* max_children) {
  if (t == nullptr) return BEAMDEC_ERR_INVALID_ARG;
  if (levels) *levels = t->levels;
  if (vocab) *vocab = t->vocab;
  if (n_distinct) *n_distinct = t->n_items;
  for (int l = 0; l < t->levels; ++l) {
    if (n_nodes) n_nodes[l] = t->n_nodes[l];
    if (n_edges) n_edges[l] = t->n_edges[l];
    if (max_children) max_children[l] = t->max_children[l];
  }
  return BEAMDEC_OK;
}

extern "C" int beam_trie_export(const beamdec_trie* t, int level, const int32_t** off,
                                const int32_t** code) {
  if (t == nullptr || level < 0 || level >= t->levels) return BEAMDEC_ERR_INVALID_ARG;
  if (off) *off = t->off[level];
  if (code) *code = t->code[level];
  return BEAMDEC_OK;
}

// Dense child masks of one level (the FlashRec announcement's fused SID trie
// has a dense and a CSR form): bit c of node n's mask is set when code c is one of
// n's children.  Built from the level's CSR (copied back to the host once);
// the CSR stays, the selection enumerates candidates from the mask.
extern "C" int beam_trie_make_dense(beamdec_trie* t, int level, void* stream_ptr) {
  if (t == nullptr || level < 0 || level >= t->levels) return BEAMDEC_ERR_INVALID_ARG;
  const int32_t C = t->C[level];
  const int64_t words = (C + 31) / 32;
  if (C > 16384 || t->n_nodes[level] * words * 4 > ((int64_t)1 << 30)) return BEAMDEC_ERR_UNSUPPORTED;
  if (t->mask[level] != nullptr) return BEAMDEC_OK;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int64_t nn = t->n_nodes[level], ne = t->n_edges[level];
  std::vector<int32_t> off(nn + 1), code(ne);
  if (cudaMemcpyAsync(off.data(), t->off[level], (nn + 1) * sizeof(int32_t), cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess ||
      cudaMemcpyAsync(code.data(), t->code[level], ne * sizeof(int32_t), cudaMemcpyDeviceToHost,
                      stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return BEAMDEC_ERR_CUDA;
  std::vector<uint32_t> mask((size_t)(nn * words), 0u);
  for (int64_t n = 0; n < nn; ++n)
    for (int32_t e = off[n]; e < off[n + 1]; ++e)
      mask[n * words + code[e] / 32] |= 1u << (code[e] % 32);
  uint32_t* d = nullptr;
  if (cudaMalloc(&d, mask.size() * sizeof(uint32_t)) != cudaSuccess) return BEAMDEC_ERR_ALLOC;
  if (cudaMemcpyAsync(d, mask.data(), mask.size() * sizeof(uint32_t), cudaMemcpyHostToDevice, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaFree(d);
    return BEAMDEC_ERR_CUDA;
  }
  t->mask[level] = d;
  t->mask_words[level] = (int32_t)words;
  return BEAMDEC_OK;
}

extern "C" int beam_trie_drop_dense(beamdec_trie* t, int level) {
  if (t == nullptr || level < 0 || level >= t->levels) return BEAMDEC_ERR_INVALID_ARG;
  if (t->mask[level] != nullptr) cudaFree(t->mask[level]);
  t->mask[level] = nullptr;
  t->mask_words[level] = 0;
  return BEAMDEC_OK;
}

extern "C" int beam_trie_export_dense(const beamdec_trie* t, int level, const uint32_t** mask,
                                      int32_t* words) {
  if (t == nullptr || level < 0 || level >= t->levels) return BEAMDEC_ERR_INVALID_ARG;
  if (mask) *mask = t->mask[level];
  if (words) *words = t->mask_words[level];
  return BEAMDEC_OK;
}
