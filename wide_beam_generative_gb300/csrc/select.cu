// Beam expansion: log-softmax, catalog-trie mask, per-beam top_k and global
// top-W selection with the slot-table update.
//
// "Generative recommendation design" (xLLM) §4.1.1: each of the beam_width
// beams expands top_k candidates and beam_width beams are chosen from the
// beam_width x top_k pool; §4.3: invalid item paths are filtered before they
// become candidates, sorting stops early; §6: cache selection follows the
// reorder.  FlashRec (SGLang PR 31626 thread): fused SID trie in CSR form.
//
// One or two launches per step:
//   bd_stream_select_kernel  a few blocks per live beam row (about 32K logits
//                      each) stream the row once for its log-sum-exp; the
//                      row's last block then scores the trie children (or
//                      the whole vocabulary), keeps the row's top_k (block
//                      radix select) and appends them to the request's pool
//                      as 64-bit keys while the row is still in L2.  When a
//                      request's pool is at most 1M keys (W <= 4096), the
//                      last row of the request selects the request's top-W
//                      itself (score-bin histogram, bucket sort, outputs), so
//                      one request's tail overlaps the others' streams.
//   bd_expand_kernel   the same per-row and per-request work when the caller
//                      passes the row normalisers (lse_in): one block per row.
//   bd_global_kernel   larger pools: cooperative grid; per request, radix select of the
//                      beam_width smallest pool keys (12-bit digits, block-
//                      private histograms merged in global memory), a bitonic
//                      sort of the survivors in shared memory, then the outputs
//                      and the parent-pointer slot rows.
// The 64-bit key (desc(score) << 32 | beam << 18 | token) orders candidates
// by (score desc, beam asc, token asc), so the selection is deterministic.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "gumbel.cuh"
#include "internal.h"

namespace bd {
namespace {

constexpr int kExpandThreads = 512;
constexpr int kGlobalThreads = 512;
constexpr int kDigitBits = 12;
constexpr int kBins = 1 << kDigitBits;  // 4096
constexpr int kMaxRowSplits = 8;         // blocks that stream one logits row together
constexpr int kTailCap = 4096;          // keys one expand block can select in shared memory

struct SelState {
  unsigned long long prefix;  // resolved high bits of the threshold key
  int32_t total;              // pool size of the request
  int32_t n_target;           // min(W, total)
  int32_t need;               // keys still to take inside the current prefix
  int32_t sure;               // keys strictly below the current prefix
  int32_t shift;              // bits below the resolved prefix (64 = none resolved)
  int32_t done;
  int32_t ncand;
  int32_t tickets;            // expand blocks of the request that have finished
  int32_t bin_mode;           // 1: the pool is gathered by score bin (no radix passes)
  int32_t bin_cut;            // last score bin gathered in bin mode
  uint32_t cutq;              // wide-row select: kTailBins - 1 - the tightest cut bin published (0: none)
  int32_t pad[3];
};
static_assert(sizeof(SelState) == 64, "state size");

struct SelWs {
  WsHeader* hdr;
  SelState* state;        // [R]
  int32_t* rowtick;       // [R][W] finished chunk blocks per row
  uint32_t* hist;         // [R][kBins]
  uint32_t* cuthist;      // [R][kBins] score-bin counts of the pool when the
                          // cooperative kernel selects (the fused tail keeps them in hist)
  uint32_t* seedhist;     // [R][kBins] score-bin counts of the cut seeds (open vocabulary)
  unsigned long long* pool;  // [R][W*Kp]
  unsigned long long* cand;  // [R][kSelectCap]
  float2* rowpart;        // [R][W][kMaxRowSplits] per-chunk (max, sum of exp)
  float* rowlse;          // [R][W] row log-sum-exp (Gumbel mode: the outputs recompute scores)
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

__host__ __device__ inline SelWs carve(void* ws, int R, int W, int Kp) {
  char* p = (char*)ws;
  SelWs s;
  s.hdr = (WsHeader*)p; p += kWsHeaderBytes;
  s.state = (SelState*)p; p += align256((size_t)R * sizeof(SelState));
  s.rowtick = (int32_t*)p; p += align256((size_t)R * W * sizeof(int32_t));
  s.hist = (uint32_t*)p; p += align256((size_t)R * kBins * sizeof(uint32_t));
  s.cuthist = (uint32_t*)p; p += align256((size_t)R * kBins * sizeof(uint32_t));
  s.seedhist = (uint32_t*)p; p += align256((size_t)R * kBins * sizeof(uint32_t));
  s.pool = (unsigned long long*)p; p += align256((size_t)R * W * Kp * 8);
  s.cand = (unsigned long long*)p; p += align256((size_t)R * kSelectCap * 8);
  s.rowpart = (float2*)p; p += align256((size_t)R * W * kMaxRowSplits * sizeof(float2));
  s.rowlse = (float*)p;
  return s;
}

// One warp: find the digit bin D holding the `need`-th smallest key (1-based)
// of a histogram; returns D and the count of keys in bins below D.
__device__ void warp_find_digit(const volatile uint32_t* hist, int nbins, uint32_t need,
                                uint32_t* D, uint32_t* below) {
  const int lane = threadIdx.x & 31;
  const int per = nbins / 32;   // a power of two
  uint32_t sum = 0;
  // lane l sums bins [l*per, (l+1)*per) starting at offset l: when per is a
  // multiple of 32 the 32 lanes of one load hit 32 different banks
  for (int i = 0; i < per; ++i) sum += hist[lane * per + ((i + lane) & (per - 1))];
  uint32_t incl = sum;
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  uint32_t excl = incl - sum;
  unsigned hit = __ballot_sync(0xffffffffu, excl < need && need <= incl);
  int src = __ffs(hit) - 1;   // exactly one lane holds the need-th key
  if (lane == src) {
    uint32_t c = excl;
    int d = lane * per;
    for (int i = 0; i < per; ++i) {
      uint32_t h = hist[lane * per + i];
      if (c + h >= need) { d = lane * per + i; break; }
      c += h;
    }
    *D = (uint32_t)d;
    *below = c;
  }
  __syncwarp();
}

// The digit holding the need-th smallest key (need >= 1) of a shared-memory
// histogram of nb digits (a power of two, at most 4 * kExpandThreads),
// searched by the whole block: thread t sums its nb / kExpandThreads
// consecutive digits (one digit, or none, when nb is smaller), one block
// prefix sum places them, and the thread whose digits hold the need-th key
// walks them again and writes sh.digit = that digit and sh.below = keys in lower digits.  A
// histogram of fewer than need keys is searched for its last key (none: digit
// 0, below 0).  Every thread of a kExpandThreads block calls it; it ends with
// a block barrier.  (One warp scanning 2048 digits alone is a serial chain of
// 64 shared loads per lane: about 2 us per radix pass.)  Not inlined: inside
// the 32-register stream kernels it would crowd the callers' registers.
template <class Smem>
__device__ __noinline__ void block_find_digit(const uint32_t* h, int nb, uint32_t need, Smem& sh) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int per = nb > kExpandThreads ? nb / kExpandThreads : 1;
  const int d0 = t * per;
  const bool mine = d0 < nb;   // digits d0 .. d0 + per - 1 are this thread's
  uint32_t sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) sum += (i < per && mine) ? h[d0 + i] : 0u;
  uint32_t inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sh.warp_cnt[warp] = (int)inc;
  __syncthreads();
  uint32_t run = inc - sum, tot = 0;
  for (int w = 0; w < kExpandThreads / 32; ++w) {
    const uint32_t c = (uint32_t)sh.warp_cnt[w];
    if (w < warp) run += c;
    tot += c;
  }
  if (need > tot) need = tot;
  if (t == 0 && tot == 0) {
    sh.digit = 0;
    sh.below = 0;
  }
  if (mine && run < need && need <= run + sum) {   // the need-th key is in this thread's digits
    for (int j = 0; j < per; ++j) {
      const uint32_t c = h[d0 + j];
      if (need <= run + c) {
        sh.digit = (uint32_t)(d0 + j);
        sh.below = run;
        break;
      }
      run += c;
    }
  }
  __syncthreads();
}

// Block-wide exclusive rank of `flag` among the block's threads, and the total.
__device__ __forceinline__ int block_rank(int flag, int* warp_cnt, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  unsigned bal = __ballot_sync(0xffffffffu, flag);
  int r = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) warp_cnt[warp] = __popc(bal);
  __syncthreads();
  int base = 0, tot = 0;
  for (int w = 0; w < nw; ++w) {
    int c = warp_cnt[w];
    if (w < warp) base += c;
    tot += c;
  }
  __syncthreads();
  *total = tot;
  return base + r;
}

// Block-wide exclusive prefix sum of v over the block's threads, and the total.
__device__ __forceinline__ int block_excl_sum(int v, int* warp_cnt, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) warp_cnt[warp] = inc;
  __syncthreads();
  int base = 0, tot = 0;
  for (int w = 0; w < nw; ++w) {
    const int c = warp_cnt[w];
    if (w < warp) base += c;
    tot += c;
  }
  __syncthreads();
  *total = tot;
  return base + inc - v;
}

// Adds one to hist[bin] for every lane with `on`: lanes that share a bin add
// their count once, so a histogram whose keys crowd into a few bins costs one
// atomic per bin and warp instead of one per key.  Every lane of the warp
// calls it (shared or global memory).
__device__ __forceinline__ void warp_hist_add(uint32_t* hist, uint32_t bin, bool on) {
  const unsigned act = __ballot_sync(0xffffffffu, on);
  if (on) {
    const unsigned peers = __match_any_sync(act, bin);
    if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(hist + bin, (uint32_t)__popc(peers));
  }
}

// Reserves one slot of *counter for every lane with `on` (one atomic per
// warp) and returns this lane's slot (unordered across warps).  Every lane of
// the warp calls it.
__device__ __forceinline__ int warp_reserve(int* counter, bool on) {
  const unsigned act = __ballot_sync(0xffffffffu, on);
  const int lane = threadIdx.x & 31;
  const int leader = act ? __ffs(act) - 1 : 0;
  int base = 0;
  if (act && lane == leader) base = atomicAdd(counter, __popc(act));
  base = __shfl_sync(0xffffffffu, base, leader);
  return base + __popc(act & ((1u << lane) - 1u));
}

// Reserves one slot of cursor[bin] for every lane with `on`; lanes that share
// a bin take consecutive slots with one atomic.  Every lane of the warp calls
// it; lanes without `on` get 0.
__device__ __forceinline__ uint32_t warp_bin_reserve(uint32_t* cursor, uint32_t bin, bool on) {
  const unsigned act = __ballot_sync(0xffffffffu, on);
  const int lane = threadIdx.x & 31;
  uint32_t base = 0;
  int leader = 0;
  unsigned peers = 0;
  if (on) {
    peers = __match_any_sync(act, bin);
    leader = __ffs(peers) - 1;
    if (lane == leader) base = atomicAdd(cursor + bin, (uint32_t)__popc(peers));
  }
  base = __shfl_sync(0xffffffffu, base, leader);
  return on ? base + (uint32_t)__popc(peers & ((1u << lane) - 1u)) : 0u;
}

// Coarse bin of a candidate score relative to a per-request reference score
// (the score of the request's rank-0 beam): floor((ref - s) * 64), clamped to
// [0, 4095].  It is monotone (a higher score never gets a higher bin), so a
// request-wide histogram of bins brackets the W-th best score from one count.
constexpr int kTailBins = 4096;
constexpr int kKeyCache = 8192;   // children whose 32-bit keys a block caches in shared memory
__device__ __forceinline__ int score_bin(float ref, float s) {
  const float u = __fmul_rn(__fsub_rn(ref, s), 64.f);
  if (!(u > 0.f)) return 0;
  if (u >= (float)(kTailBins - 1)) return kTailBins - 1;
  return (int)u;
}

// Reference of the score bins: the request's rank-0 cumulative score, or in
// Gumbel mode (kG) its ordering-key scale plus 16 (a Gumbel draw exceeds 16
// with probability 1e-7; keys above the reference all land in bin 0).
template <bool kG>
__device__ __forceinline__ float bin_ref(const SelectArgs& a, float cum0) {
  return kG ? __fadd_rn(__fmul_rn(cum0, a.inv_tau), 16.f) : cum0;
}

struct ExpandShared {
  uint32_t hist[2048];
  float red_m[32];
  float red_s[32];
  int warp_cnt[32];
  uint32_t digit, below;
  int count;
  int pool_base;
  int cnt2, cnt3;   // slot counters of the wide-row path
  float lse;
  uint32_t c_le;
  // the row's trie range and score, fetched at the start of a stream block
  // so that the row's expansion does not wait on them (pf_e0 < 0: not fetched)
  int pf_e0, pf_e1;
  float pf_cum, pf_ref;
};

// Running (max, sum of exp(x - max)) of row[c0..c1) for the whole block,
// returned to every thread.  One streaming pass: four 16-byte loads in
// flight per thread, the exponentials with the ex2 instruction.
__device__ __forceinline__ float2 stream_max_sum(const float* row, int c0, int c1, ExpandShared& sh) {
  const int tid = threadIdx.x;
  float m = -INFINITY, s = 0.f;
  const float* base = row + c0;
  const int len = c1 - c0;
  const bool vec = ((reinterpret_cast<uintptr_t>(base) & 15u) == 0);
  const int nvec = vec ? (len >> 2) : 0;
  const float4* row4 = reinterpret_cast<const float4*>(base);
  int i = tid;
  for (; i + 3 * kExpandThreads < nvec; i += 4 * kExpandThreads) {
    float4 v0 = __ldg(row4 + i);
    float4 v1 = __ldg(row4 + i + kExpandThreads);
    float4 v2 = __ldg(row4 + i + 2 * kExpandThreads);
    float4 v3 = __ldg(row4 + i + 3 * kExpandThreads);
    float mx = fmaxf(fmaxf(fmaxf(v0.x, v0.y), fmaxf(v0.z, v0.w)),
                     fmaxf(fmaxf(v1.x, v1.y), fmaxf(v1.z, v1.w)));
    mx = fmaxf(mx, fmaxf(fmaxf(fmaxf(v2.x, v2.y), fmaxf(v2.z, v2.w)),
                         fmaxf(fmaxf(v3.x, v3.y), fmaxf(v3.z, v3.w))));
    if (mx > m) { s *= ex2((m - mx) * kLog2e); m = mx; }
    const float mL = m * kLog2e;
    float t0 = ex2(fmaf(v0.x, kLog2e, -mL)) + ex2(fmaf(v0.y, kLog2e, -mL)) +
               ex2(fmaf(v0.z, kLog2e, -mL)) + ex2(fmaf(v0.w, kLog2e, -mL));
    float t1 = ex2(fmaf(v1.x, kLog2e, -mL)) + ex2(fmaf(v1.y, kLog2e, -mL)) +
               ex2(fmaf(v1.z, kLog2e, -mL)) + ex2(fmaf(v1.w, kLog2e, -mL));
    float t2 = ex2(fmaf(v2.x, kLog2e, -mL)) + ex2(fmaf(v2.y, kLog2e, -mL)) +
               ex2(fmaf(v2.z, kLog2e, -mL)) + ex2(fmaf(v2.w, kLog2e, -mL));
    float t3 = ex2(fmaf(v3.x, kLog2e, -mL)) + ex2(fmaf(v3.y, kLog2e, -mL)) +
               ex2(fmaf(v3.z, kLog2e, -mL)) + ex2(fmaf(v3.w, kLog2e, -mL));
    s += (t0 + t1) + (t2 + t3);
  }
  for (; i < nvec; i += kExpandThreads) {
    float4 v = __ldg(row4 + i);
    float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
    if (mx > m) { s *= ex2((m - mx) * kLog2e); m = mx; }
    const float mL = m * kLog2e;
    s += ex2(fmaf(v.x, kLog2e, -mL)) + ex2(fmaf(v.y, kLog2e, -mL)) +
         ex2(fmaf(v.z, kLog2e, -mL)) + ex2(fmaf(v.w, kLog2e, -mL));
  }
  for (int j = nvec * 4 + tid; j < len; j += kExpandThreads) {
    float x = __ldg(base + j);
    if (x > m) { s *= ex2((m - x) * kLog2e); m = x; }
    s += ex2((x - m) * kLog2e);
  }
  // block reduction of (m, s)
  for (int o = 16; o; o >>= 1) {
    float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    float M = fmaxf(m, m2);
    float a1 = (s == 0.f) ? 0.f : s * ex2((m - M) * kLog2e);
    float a2 = (s2 == 0.f) ? 0.f : s2 * ex2((m2 - M) * kLog2e);
    m = M; s = a1 + a2;
  }
  const int lane = tid & 31, warp = tid >> 5;
  if (lane == 0) { sh.red_m[warp] = m; sh.red_s[warp] = s; }
  __syncthreads();
  if (warp == 0) {
    const int nw = kExpandThreads / 32;
    m = lane < nw ? sh.red_m[lane] : -INFINITY;
    s = lane < nw ? sh.red_s[lane] : 0.f;
    for (int o = 16; o; o >>= 1) {
      float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      float M = fmaxf(m, m2);
      float a1 = (s == 0.f) ? 0.f : s * ex2((m - M) * kLog2e);
      float a2 = (s2 == 0.f) ? 0.f : s2 * ex2((m2 - M) * kLog2e);
      m = M; s = a1 + a2;
    }
    if (lane == 0) { sh.red_m[0] = m; sh.red_s[0] = s; }
  }
  __syncthreads();
  const float2 res = make_float2(sh.red_m[0], sh.red_s[0]);
  __syncthreads();
  return res;
}


// Rows a2-a3 for beam b of request r: log-sum-exp, trie children, per-beam
// top_k appended to the request's pool.
// gh (the request's score-bin histogram in global memory; fused launches
// only) counts every candidate the row adds to the pool.
// kPf: the row's trie range and scores were fetched into sh.pf_* already.
// kG: Gumbel top-k; candidates are ordered by fl32(fl32(s * inv_tau) + g).
// kD: the level has dense child masks; candidates are enumerated from the
//     node's mask (bit order = code order = child order) instead of its CSR
//     code list.  Built into the expansion kernel only (lse_in given): the
//     32-register stream kernel keeps the CSR enumeration.
// Ordering key of a candidate of beam b (request r) with logit x and token
// tok: s = fl32(cum + fl32(x - lse)), or with kG the Gumbel key
// fl32(fl32(s * inv_tau) + g), as a 32-bit key (smaller = better).
template <bool kG>
__device__ __forceinline__ uint32_t cand_key(const SelectArgs& a, float cum, float lse, float x, int r,
                                             int b, int tok) {
  const float sc = __fadd_rn(cum, __fsub_rn(x, lse));
  if constexpr (kG)
    return desc_key(__fadd_rn(__fmul_rn(sc, a.inv_tau), gumbel_noise(a.seed_lo, a.seed_hi, r, a.step, b, tok)));
  else
    return desc_key(sc);
}

template <bool kG>
__device__ __forceinline__ bool expand_wide(const SelectArgs& a, ExpandShared& sh, SelState* st,
                                            unsigned long long* pool, uint32_t* gh, const uint32_t* seed,
                                            unsigned char* dyn, const float* row, const int32_t* code,
                                            int tb, int n, int r, int b, float cum, float lse, float ref);

template <bool kPf, bool kG, bool kD>
__device__ __forceinline__ void expand_candidates(const SelectArgs& a, ExpandShared& sh, const SelWs& ws,
                                                 int r, int b, uint32_t* gh, uint32_t* kcache,
                                                 float lse) {
  static_assert(!(kPf && kD), "dense masks are enumerated by the expansion kernel only");
  const int tid = threadIdx.x;
  const int Kp = a.Kp;
  const size_t rowi = (size_t)r * a.W + b;
  const float* row = a.logits + rowi * (size_t)a.row_stride;

  if (a.lse_in != nullptr && a.lse_out != nullptr && tid == 0) a.lse_out[rowi] = lse;
  const float cum = kPf ? sh.pf_cum : a.cum_in[rowi];

  // ---- a2: candidate range (trie children or the whole vocabulary) --------
  int n = a.V;
  const int32_t* code = nullptr;
  int tb = 0;
  int node = -1;
  if (a.has_trie) {
    int e0, e1;
    if constexpr (kPf) {
      e0 = sh.pf_e0;
      e1 = sh.pf_e1;
    } else {
      node = a.node_in[rowi];
      const bool bad = node < 0 || node >= a.lvl.n_nodes;
      e0 = bad ? -2 : a.lvl.off[node];
      e1 = bad ? -2 : a.lvl.off[node + 1];
    }
    if (e0 < 0) {
      if (tid == 0) set_status(ws.hdr, BEAMDEC_ERR_DEVICE_CHECK);
      return;
    }
    n = e1 - e0;
    code = a.lvl.code + e0;
    tb = a.lvl.token_base;
  }
  auto tok_of = [&](int i) -> int { return code ? tb + __ldg(code + i) : i; };
  // ordering key of token tok whose logit is x
  auto score_key = [&](float x, int tok) -> uint32_t { return cand_key<kG>(a, cum, lse, x, r, b, tok); };
  auto key_of = [&](int tok) -> uint32_t { return score_key(__ldg(row + tok), tok); };
  // kD: every child (index, token, key) from the node's dense mask, handed to
  // sink(on, child, key) by every thread of the block (block-uniform rounds
  // of four positions per thread; logits only for set bits)
  auto dense_children = [&](auto&& sink) {
    const int words = a.lvl.words;
    uint32_t* wsm = sh.hist;           // the node's mask words
    uint32_t* pre = sh.hist + 1024;    // children in the words before each word
    const uint32_t wv = tid < words ? __ldg(a.lvl.mask + (size_t)node * words + tid) : 0u;
    int tot;
    const int ex = block_excl_sum(__popc(wv), sh.warp_cnt, &tot);
    if (tid < words) {
      wsm[tid] = wv;
      pre[tid] = (uint32_t)ex;
    }
    __syncthreads();
    constexpr int kU = 4;
    const int C = 32 * words;
    for (int c0 = 0; c0 < C; c0 += kU * kExpandThreads) {
      bool on[kU];
      int child[kU];
      float x[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int pos = c0 + u * kExpandThreads + tid;
        const uint32_t w = pos < C ? wsm[pos >> 5] : 0u;
        on[u] = (w >> (pos & 31)) & 1u;
        child[u] = (int)pre[pos < C ? pos >> 5 : 0] + __popc(w & ((1u << (pos & 31)) - 1u));
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) x[u] = on[u] ? __ldg(row + tb + c0 + u * kExpandThreads + tid) : 0.f;
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int tok = tb + c0 + u * kExpandThreads + tid;
        sink(on[u], child[u], on[u] ? score_key(x[u], tok) : 0u);
      }
    }
  };

  SelState* st = ws.state + r;
  unsigned long long* pool = ws.pool + (size_t)r * a.W * Kp;
  const float ref = bin_ref<kG>(a, kPf ? sh.pf_ref : a.cum_in[(size_t)r * a.W]);

  // ---- a3: per-beam top_k -------------------------------------------------
  if (n <= a.K) {
    if constexpr (kD) {
      if (tid == 0) sh.pool_base = n > 0 ? atomicAdd(&st->total, n) : 0;
      __syncthreads();   // (dense_children's own barriers follow; pool_base is read after them)
      dense_children([&](bool on, int child, uint32_t k) {
        if (on) pool[sh.pool_base + child] = pool_key(k, b, child);
        if (gh) warp_hist_add(gh, (uint32_t)score_bin(ref, desc_key_value(k)), on);
      });
      return;
    }
    // the first round's gathers are in flight while the pool slots are reserved
    const uint32_t k_first = tid < n ? key_of(tok_of(tid)) : 0u;
    if (tid == 0) sh.pool_base = n > 0 ? atomicAdd(&st->total, n) : 0;
    __syncthreads();
    const int base = sh.pool_base;
    for (int c0 = 0; c0 < n; c0 += kExpandThreads) {   // block-uniform trip count
      const int i = c0 + tid;
      const bool on = i < n;
      const uint32_t k = c0 == 0 ? k_first : (on ? key_of(tok_of(i)) : 0u);
      if (on) pool[base + i] = pool_key(k, b, i);
      if (gh) warp_hist_add(gh, (uint32_t)score_bin(ref, desc_key_value(k)), on);
    }
    return;
  }
  // the row's candidate keys, computed once into shared memory when they fit
  // (the radix passes below then read shared memory instead of re-gathering)
  const bool cached = kcache != nullptr && n <= kKeyCache;
  if (kD && cached) {
    dense_children([&](bool on, int child, uint32_t k) {
      if (on) kcache[child] = k;
    });
    __syncthreads();
  } else if (cached) {   // four children per thread in flight: codes first, then their logits
    constexpr int kU = 4;
    for (int c0 = 0; c0 < n; c0 += kU * kExpandThreads) {
      int tk[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = c0 + u * kExpandThreads + tid;
        tk[u] = i < n ? tok_of(i) : 0;
      }
      float x[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) x[u] = __ldg(row + tk[u]);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = c0 + u * kExpandThreads + tid;
        if (i < n) kcache[i] = score_key(x[u], tk[u]);
      }
    }
    __syncthreads();
  }
  // more candidates than the key cache holds (the expansion kernel): two
  // passes over a score-bin histogram; the radix passes below remain the
  // exact fallback for heavy ties
  if constexpr (!kPf) {
    if (!cached && kcache != nullptr && gh != nullptr &&
        expand_wide<kG>(a, sh, st, pool, gh, a.seeded ? ws.seedhist + (size_t)r * kBins : nullptr,
                        reinterpret_cast<unsigned char*>(kcache), row, code, tb, n, r, b, cum, lse, ref))
      return;
  }
  auto kc = [&](int i) -> uint32_t { return cached ? kcache[i] : key_of(tok_of(i)); };
  // radix select of the K-th smallest 32-bit score key: digits of 11, 11, 10 bits
  uint32_t prefix = 0, need = (uint32_t)a.K;
  const int widths[3] = {11, 11, 10};
  int shift = 32;
  for (int pass = 0; pass < 3; ++pass) {
    const int w = widths[pass];
    const int nb = 1 << w;
    const int sh_next = shift - w;
    for (int i = tid; i < nb; i += kExpandThreads) sh.hist[i] = 0;
    __syncthreads();
    if (cached) {
      for (int c0 = 0; c0 < n; c0 += kExpandThreads) {   // block-uniform trip count
        const int i = c0 + tid;
        const uint32_t k = i < n ? kcache[i] : 0u;
        const bool on = i < n && (shift == 32 || (k >> shift) == (prefix >> shift));
        warp_hist_add(sh.hist, (k >> sh_next) & (nb - 1), on);
      }
    } else {   // keys from the row again: four logits per thread in flight
      for (int c0 = 0; c0 < n; c0 += 4 * kExpandThreads) {   // block-uniform trip count
        float x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = c0 + u * kExpandThreads + tid;
          x[u] = i < n ? __ldg(row + tok_of(i)) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = c0 + u * kExpandThreads + tid;
          const uint32_t k = i < n ? score_key(x[u], tok_of(i)) : 0u;
          const bool on = i < n && (shift == 32 || (k >> shift) == (prefix >> shift));
          warp_hist_add(sh.hist, (k >> sh_next) & (nb - 1), on);
        }
      }
    }
    __syncthreads();
    block_find_digit(sh.hist, nb, need, sh);
    prefix |= sh.digit << sh_next;
    need -= sh.below;
    shift = sh_next;
    __syncthreads();
  }
  const uint32_t kth = prefix;   // exact K-th smallest key; `need` ties at kth are kept
  if (tid == 0) { sh.count = 0; sh.pool_base = atomicAdd(&st->total, a.K); }
  __syncthreads();
  const int base = sh.pool_base;
  auto take_below = [&](int i, uint32_t k) {   // every key below the K-th goes to the pool
    const bool on = i < n && k < kth;
    const int pos = warp_reserve(&sh.count, on);
    if (on) pool[base + pos] = pool_key(k, b, i);
    if (gh) warp_hist_add(gh, (uint32_t)score_bin(ref, desc_key_value(k)), on);
  };
  if (cached) {
    for (int c0 = 0; c0 < n; c0 += kExpandThreads) {   // block-uniform trip count
      const int i = c0 + tid;
      take_below(i, i < n ? kcache[i] : 0u);
    }
  } else {   // four logits per thread in flight, as in the radix passes
    for (int c0 = 0; c0 < n; c0 += 4 * kExpandThreads) {   // block-uniform trip count
      float x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = c0 + u * kExpandThreads + tid;
        x[u] = i < n ? __ldg(row + tok_of(i)) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = c0 + u * kExpandThreads + tid;
        take_below(i, i < n ? score_key(x[u], tok_of(i)) : 0u);
      }
    }
  }
  __syncthreads();
  const int n_less = sh.count;
  int taken = 0;
  for (int c0 = 0; c0 < n && taken < (int)need; c0 += kExpandThreads) {
    const int i = c0 + tid;
    int flag = 0;
    if (i < n) flag = kc(i) == kth;
    int tot;
    const int rk = block_rank(flag, sh.warp_cnt, &tot);
    const bool on = flag && taken + rk < (int)need;
    if (on) pool[base + n_less + taken + rk] = pool_key(kth, b, i);
    if (gh) warp_hist_add(gh, (uint32_t)score_bin(ref, desc_key_value(kth)), on);
    taken += tot;
  }
}

// Ascending bitonic sort of np (a power of two) 64-bit keys in shared memory.
__device__ void bitonic_sort(unsigned long long* keys, int np) {
  for (int k = 2; k <= np; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < np; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long x = keys[i], y = keys[ixj];
          const bool up = (i & k) == 0;
          if ((x > y) == up) { keys[i] = y; keys[ixj] = x; }
        }
      }
      __syncthreads();
    }
  }
}

// a4/a5 outputs of request r from its nt winners, sorted ascending in keys[]:
// tokens, parents, scores, child nodes, live count and the slot rows
// (parent's row up to step-1, then step*W + j).
// poff (optional): poff[j] = first edge of live beam j's trie node, gathered
// earlier so the decode waits on one load instead of three.
// kG: the pool keys hold the noisy ordering key, so the returned score is
// recomputed from the parent's row: fl32(cum + fl32(logit - lse)).
template <bool kG>
__device__ void emit_outputs(const SelectArgs& a, const SelWs& ws, int r,
                             const unsigned long long* keys, int nt, const int* poff = nullptr) {
  const int tid = threadIdx.x;
  const size_t o = (size_t)r * a.W;
  for (int j = tid; j < a.W; j += blockDim.x) {
    if (j < nt) {
      const unsigned long long k = keys[j];
      const int parent = pool_key_beam(k), idx = pool_key_tok(k);
      int tok = idx, node = -1;
      if (a.has_trie) {
        node = (poff ? poff[parent] : a.lvl.off[a.node_in[o + parent]]) + idx;   // edge index = child node
        tok = a.lvl.token_base + a.lvl.code[node];
      }
      a.tokens[o + j] = tok;
      a.parents[o + j] = parent;
      if constexpr (kG) {
        const size_t pr = o + parent;
        const float lse = a.lse_in != nullptr ? a.lse_in[pr] : __ldcg(ws.rowlse + pr);
        const float x = a.logits[pr * (size_t)a.row_stride + tok];
        a.cum_out[o + j] = __fadd_rn(a.cum_in[pr], __fsub_rn(x, lse));
      } else {
        a.cum_out[o + j] = desc_key_value((uint32_t)(k >> 32));
      }
      a.node_out[o + j] = node;
    } else {
      a.tokens[o + j] = -1;
      a.parents[o + j] = -1;
      a.cum_out[o + j] = -INFINITY;
      a.node_out[o + j] = -1;
    }
  }
  const int T = a.T;
  for (int idx = tid; idx < a.W * T; idx += blockDim.x) {
    const int j = idx / T, t = idx - j * T;
    int v = -1;
    if (j < nt) {
      if (t < a.step) v = a.slot_in[(o + pool_key_beam(keys[j])) * T + t];
      else if (t == a.step) v = a.step * a.W + j;
    }
    a.slot_out[(o + j) * T + t] = v;
  }
  if (tid == 0) a.n_live_out[r] = nt;
}

// Output row j < n_target of request r for pool key k, as emit_outputs
// writes it, by a group of eight threads (part 0..7): part 0 the token,
// parent, score and node, the eight together the slot row.
template <bool kG>
__device__ __forceinline__ void emit_row(const SelectArgs& a, const SelWs& ws, int r, int j,
                                         unsigned long long k, int part) {
  const size_t o = (size_t)r * a.W;
  const int parent = pool_key_beam(k);
  if (part == 0) {
    const int idx = pool_key_tok(k);
    int tok = idx, node = -1;
    if (a.has_trie) {
      node = a.lvl.off[a.node_in[o + parent]] + idx;   // edge index = child node
      tok = a.lvl.token_base + a.lvl.code[node];
    }
    a.tokens[o + j] = tok;
    a.parents[o + j] = parent;
    if constexpr (kG) {
      const size_t pr = o + parent;
      const float lse = a.lse_in != nullptr ? a.lse_in[pr] : __ldcg(ws.rowlse + pr);
      const float x = a.logits[pr * (size_t)a.row_stride + tok];
      a.cum_out[o + j] = __fadd_rn(a.cum_in[pr], __fsub_rn(x, lse));
    } else {
      a.cum_out[o + j] = desc_key_value((uint32_t)(k >> 32));
    }
    a.node_out[o + j] = node;
  }
  const int T = a.T;
  for (int t = part; t < T; t += 8) {
    int v = -1;
    if (t < a.step) v = a.slot_in[(o + parent) * T + t];
    else if (t == a.step) v = a.step * a.W + j;
    a.slot_out[(o + j) * T + t] = v;
  }
}

// Output row j >= n_target of request r (a dead beam), as emit_outputs writes it.
__device__ __forceinline__ void emit_dead_row(const SelectArgs& a, int r, int j) {
  const size_t o = (size_t)r * a.W;
  a.tokens[o + j] = -1;
  a.parents[o + j] = -1;
  a.cum_out[o + j] = -INFINITY;
  a.node_out[o + j] = -1;
  for (int t = 0; t < a.T; ++t) a.slot_out[(o + j) * a.T + t] = -1;
}

// Sorts keys[0..n) ascending in place, n <= 2 * kExpandThreads, called by
// every thread of a kExpandThreads-thread block.  A bitonic network over
// 2 * kExpandThreads slots held in registers, slots t and t + kExpandThreads
// by thread t: partners closer than 32 slots are exchanged by warp shuffles,
// farther ones through keys[] itself.  Pad slots hold ~0, above every pool
// key (bit 31 of a pool key is always 0), so they sort last.
__device__ void block_sort_small(unsigned long long* keys, int n) {
  constexpr int kH = kExpandThreads;
  const int t = threadIdx.x;
  unsigned long long x0 = t < n ? keys[t] : ~0ull;
  unsigned long long x1 = t + kH < n ? keys[t + kH] : ~0ull;
  __syncthreads();   // every read above precedes the exchange writes below
  for (int k = 2; k <= 2 * kH; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j == kH) {   // k == 2 kH: both slots of the thread, ascending
        const unsigned long long lo = x0 < x1 ? x0 : x1, hi = x0 < x1 ? x1 : x0;
        x0 = lo;
        x1 = hi;
        continue;
      }
      unsigned long long y0, y1;
      if (j >= 32) {
        keys[t] = x0;
        keys[t + kH] = x1;
        __syncthreads();
        y0 = keys[t ^ j];
        y1 = keys[(t + kH) ^ j];   // == keys[(t ^ j) + kH]: j < kH leaves that bit alone
        __syncthreads();
      } else {
        y0 = __shfl_xor_sync(0xffffffffu, x0, j);
        y1 = __shfl_xor_sync(0xffffffffu, x1, j);
      }
      // slot s keeps the smaller of its pair when it is the lower slot of an
      // ascending run or the upper slot of a descending one
      const bool min0 = ((t & j) == 0) == ((t & k) == 0);
      const bool min1 = (((t + kH) & j) == 0) == (((t + kH) & k) == 0);
      x0 = min0 ? (x0 < y0 ? x0 : y0) : (x0 < y0 ? y0 : x0);
      x1 = min1 ? (x1 < y1 ? x1 : y1) : (x1 < y1 ? y1 : x1);
    }
  }
  keys[t] = x0;
  keys[t + kH] = x1;
  __syncthreads();
}

// One radix-narrowing pass over `n` keys (shared or global memory): among the
// keys whose bits above `shift` equal `prefix`, histogram the next `w` bits
// and pick the digit holding the need-th smallest key.  Updates prefix,
// shift, need and sure (keys strictly below the new prefix); returns the
// count of keys inside the chosen digit.
template <bool kGlobal>
__device__ uint32_t narrow_pass(const unsigned long long* keys, int n, unsigned long long& prefix,
                                int& shift, uint32_t& need, uint32_t& sure, ExpandShared& sh) {
  const int w = shift < 11 ? shift : 11;
  const int nshift = shift - w;
  const uint32_t mask = (1u << w) - 1u;
  const int nb = (1 << w) < 32 ? 32 : (1 << w);
  for (int i = threadIdx.x; i < nb; i += blockDim.x) sh.hist[i] = 0;
  __syncthreads();
  for (int c0 = 0; c0 < n; c0 += blockDim.x) {   // block-uniform trip count
    const int i = c0 + threadIdx.x;
    const unsigned long long k = i < n ? (kGlobal ? __ldcg(keys + i) : keys[i]) : 0ull;
    const bool on = i < n && (shift == 64 || (k >> shift) == prefix);
    warp_hist_add(sh.hist, (uint32_t)(k >> nshift) & mask, on);
  }
  __syncthreads();
  block_find_digit(sh.hist, nb, need, sh);
  const uint32_t D = sh.digit, below = sh.below, in_bin = sh.hist[D];
  __syncthreads();
  sure += below;
  need -= below;
  prefix = (shift == 64 ? 0ull : (prefix << w)) | D;
  shift = nshift;
  return in_bin;
}

// Exclusive prefix sum of the kTailBins bins of the global histogram gh into
// hs (kExpandThreads threads, 8 bins each), and the bin holding the need-th
// key (1-based, need <= sum of all bins): sh.digit = that bin, sh.below =
// keys in lower bins, sh.c_le = keys in it and below.
__device__ void block_scan_bins(const uint32_t* gh, uint32_t* hs, uint32_t need, ExpandShared& sh) {
  constexpr int kPer = kTailBins / kExpandThreads;
  static_assert(kPer * kExpandThreads == kTailBins, "bins per thread");
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) { sh.digit = kTailBins - 1; sh.below = 0; sh.c_le = 0; }
  uint32_t v[kPer];
  uint32_t sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    v[i] = __ldcg(gh + t * kPer + i);
    sum += v[i];
  }
  uint32_t inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sh.warp_cnt[warp] = (int)inc;
  __syncthreads();
  uint32_t run = inc - sum;
  for (int w = 0; w < warp; ++w) run += (uint32_t)sh.warp_cnt[w];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const uint32_t c = v[j];
    if (run < need && need <= run + c) {
      sh.digit = (uint32_t)(t * kPer + j);
      sh.below = run;
      sh.c_le = run + c;
    }
    hs[t * kPer + j] = run;
    run += c;
  }
  __syncthreads();
}

// The bin holding the need-th key (need >= 1) of a shared-memory histogram of
// kTailBins bins: sh.digit = that bin and sh.below = keys in lower bins, or,
// when the histogram holds fewer than need keys, sh.digit = kTailBins and
// sh.below = all of them.  Every thread of a kExpandThreads block calls it.
__device__ void block_find_bin_smem(const uint32_t* h, uint32_t need, ExpandShared& sh) {
  constexpr int kPer = kTailBins / kExpandThreads;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t v[kPer];
  uint32_t sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    v[i] = h[t * kPer + i];
    sum += v[i];
  }
  uint32_t inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) sh.warp_cnt[warp] = (int)inc;
  __syncthreads();
  uint32_t run = inc - sum, tot = 0;
  for (int w = 0; w < kExpandThreads / 32; ++w) {
    const uint32_t c = (uint32_t)sh.warp_cnt[w];
    if (w < warp) run += c;
    tot += c;
  }
  if (t == 0 && tot < need) {
    sh.digit = kTailBins;
    sh.below = tot;
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const uint32_t c = v[j];
    if (run < need && need <= run + c) {
      sh.digit = (uint32_t)(t * kPer + j);
      sh.below = run;
    }
    run += c;
  }
  __syncthreads();
}

// Moves the nt smallest of the nc distinct 64-bit keys in shared memory to
// keys[0..nt) (in no particular order), 0 < nt < nc.
__device__ void smem_take_smallest(unsigned long long* keys, int nc, int nt, ExpandShared& sh) {
  if (nc <= 2 * kExpandThreads) {   // sorted ascending: the first nt are the smallest
    block_sort_small(keys, nc);
    return;
  }
  unsigned long long prefix = 0;
  int shift = 64;
  uint32_t need = (uint32_t)nt, sure = 0;
  while (true) {
    const uint32_t in_bin = narrow_pass<false>(keys, nc, prefix, shift, need, sure, sh);
    if (sure + in_bin == (uint32_t)nt || shift == 0) break;
  }
  if (threadIdx.x == 0) sh.count = 0;
  __syncthreads();
  for (int c0 = 0; c0 < nc; c0 += blockDim.x) {   // block-uniform trip count
    const int i = c0 + threadIdx.x;
    unsigned long long k = 0;
    int flag = 0;
    if (i < nc) {
      k = keys[i];
      flag = (k >> shift) <= prefix;
    }
    int tot;
    const int rk = block_rank(flag, sh.warp_cnt, &tot);   // all reads of the chunk precede writes
    if (flag) keys[sh.count + rk] = k;
    __syncthreads();
    if (threadIdx.x == 0) sh.count += tot;
    __syncthreads();
  }
}

// Per-beam top_k of a row with more candidates than the key cache holds (the
// open vocabulary; trie nodes above kKeyCache children), in the expansion
// kernel.  The row is read in block-uniform rounds (eight 16-byte loads in
// flight per thread for a contiguous row); a round in which no lane of a warp
// holds a logit above the pass's lower bound costs one vote, and the warp
// stages the logits above it in shared memory and scores them 32 at a time:
//   the request's cut: gh counts every candidate already in the request's
//     pool by score bin (bins of 1/64 below the rank-0 beam's score, so a
//     higher score never has a higher bin); once W of them lie at or above
//     bin b*, a candidate in a later bin ranks below W pool members and can
//     never be selected, so it is not emitted (the candidates that pass form
//     a prefix of the row's order, and the row's top_k among them is its
//     top_k restricted to them);
//   a counting pass, only while the request has no cut: per-thread counts,
//     over a leading part of the row, of the logits that reach each bin of a
//     ladder give a bin at or above which the row holds K candidates; it cuts
//     the row the same way;
//   pass 1: a shared-memory histogram of the passing candidates' bins; the
//     first kWideBuf of them are also buffered, and when that is all of
//     them the top_k is taken from the buffer;
//   pass 2 (otherwise): the histogram gives the bin D holding the top_k-th
//     candidate; those in bins below D go to the pool, those in bin D to the
//     buffer, of which the smallest (key, index) complete the top_k.
// The emitted candidates' bins reach gh once per bin at the end of the row.
// Returns false, having emitted nothing, when bin D holds more than kWideBuf
// candidates (heavy ties); the caller then runs the radix passes.
// dyn: the 32 KB dynamic buffer (histogram in the lower 16 KB, candidates in
// the upper 16 KB); sh.hist holds the warps' staged logits during a pass.
constexpr int kWideBuf = 2048;   // (key << 32 | index) entries
constexpr int kCutScanEvery = 16;  // rows between two scans of the pool's bin counts
// Bins of the counting ladder, counted from the bin of the beam's own score:
// 1.5 to 24 nats below it (64 bins per nat).
constexpr int kLadder = 12;
__host__ __device__ constexpr int ladder_bins(int j) {
  return j == 0 ? 96 : j == 1 ? 128 : j == 2 ? 192 : j == 3 ? 256 : j == 4 ? 320 : j == 5 ? 384
       : j == 6 ? 448 : j == 7 ? 512 : j == 8 ? 640 : j == 9 ? 768 : j == 10 ? 1024 : 1536;
}
// Adds to the request's cut histogram the bins of a row's emitted candidates:
// every candidate lh counts below bin D, and extra of bin D (one atomic per
// occupied bin, not one per candidate: the rows of a request share the few
// bins near its cut).
__device__ __forceinline__ void add_cut_hist(uint32_t* gh, const uint32_t* lh, int D, uint32_t extra) {
  for (int i = threadIdx.x; i < kTailBins; i += kExpandThreads) {
    const uint32_t c = i < D ? lh[i] : (i == D ? extra : 0u);
    if (c != 0u) atomicAdd(gh + i, c);
  }
}
template <bool kG>
__device__ __forceinline__ bool expand_wide(const SelectArgs& a, ExpandShared& sh, SelState* st,
                                            unsigned long long* pool, uint32_t* gh, const uint32_t* seed,
                                            unsigned char* dyn, const float* row, const int32_t* code,
                                            int tb, int n, int r, int b, float cum, float lse, float ref) {
  static_assert(kTailBins * 4 + kWideBuf * 8 <= kTailCap * 8, "wide-row buffers");
  static_assert(kExpandThreads / 32 * 128 <= 2048, "64 staged pairs per warp in sh.hist");
  static_assert(kLadder <= 32, "ladder counts in sh.warp_cnt");
  const int tid = threadIdx.x, lane = tid & 31;
  const int K = a.K;
  uint32_t* lh = reinterpret_cast<uint32_t*>(dyn);
  unsigned long long* buf = reinterpret_cast<unsigned long long*>(dyn + kTailBins * 4);
  float* stx = reinterpret_cast<float*>(sh.hist) + (tid >> 5) * 128;   // staged logits
  int* sti = reinterpret_cast<int*>(sh.hist) + (tid >> 5) * 128 + 64;  // and their indices
  const bool vec = code == nullptr && (reinterpret_cast<uintptr_t>(row) & 15u) == 0;
  // fn(keep, index, token, logit) for every candidate, by all lanes of a warp,
  // in the rounds where some lane of the warp keeps one (keep: not below lo)
  auto rounds = [&](float lo, auto&& fn) {
    if (vec) {
      constexpr int kV = 8;   // 16-byte loads in flight per thread
      const int nv = n >> 2;
      const float4* r4 = reinterpret_cast<const float4*>(row);
      for (int g0 = 0; g0 < nv; g0 += kV * kExpandThreads) {   // block-uniform trip count
        float4 v[kV];
#pragma unroll
        for (int u = 0; u < kV; ++u) {
          const int g = g0 + u * kExpandThreads + tid;
          v[u] = g < nv ? __ldg(r4 + g) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
        bool any = false;
#pragma unroll
        for (int u = 0; u < kV; ++u)
          any |= !(v[u].x < lo) | !(v[u].y < lo) | !(v[u].z < lo) | !(v[u].w < lo);
        if (!__any_sync(0xffffffffu, any)) continue;
#pragma unroll
        for (int u = 0; u < kV; ++u) {
          const int g = g0 + u * kExpandThreads + tid;
          const bool on = g < nv;
          fn(on && !(v[u].x < lo), 4 * g, 4 * g, v[u].x);
          fn(on && !(v[u].y < lo), 4 * g + 1, 4 * g + 1, v[u].y);
          fn(on && !(v[u].z < lo), 4 * g + 2, 4 * g + 2, v[u].z);
          fn(on && !(v[u].w < lo), 4 * g + 3, 4 * g + 3, v[u].w);
        }
      }
      for (int c0 = nv * 4; c0 < n; c0 += kExpandThreads) {   // the last n % 4 candidates
        const int i = c0 + tid;
        const float x = i < n ? __ldg(row + i) : 0.f;
        const bool keep = i < n && !(x < lo);
        if (__any_sync(0xffffffffu, keep)) fn(keep, i, i, x);
      }
    } else {
      for (int c0 = 0; c0 < n; c0 += 4 * kExpandThreads) {   // block-uniform trip count
        int tk[4];
        float x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = c0 + u * kExpandThreads + tid;
          tk[u] = i < n ? (code ? tb + __ldg(code + i) : i) : 0;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = (c0 + u * kExpandThreads + tid < n) ? __ldg(row + tk[u]) : 0.f;
        bool keep[4], any = false;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          keep[u] = c0 + u * kExpandThreads + tid < n && !(x[u] < lo);
          any |= keep[u];
        }
        if (!__any_sync(0xffffffffu, any)) continue;
#pragma unroll
        for (int u = 0; u < 4; ++u) fn(keep[u], c0 + u * kExpandThreads + tid, tk[u], x[u]);
      }
    }
  };
  // Staging (deterministic keys only: their token is not needed): the warp's
  // kept (logit, index) pairs queue in its 64 shared slots, and heavy(on,
  // index, token, logit) scores them when 32 are queued.
  int queued = 0;   // warp-uniform
  auto stage = [&](bool keep, int i, float x, auto&& heavy) {
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (m == 0u) return;
    if (keep) {
      const int p = queued + __popc(m & ((1u << lane) - 1u));
      stx[p] = x;
      sti[p] = i;
    }
    queued += __popc(m);
    if (queued >= 32) {
      __syncwarp();
      const float xs = stx[lane];
      const int is = sti[lane];
      const int rest = queued - 32;
      if (lane < rest) {   // the overflow moves to the front (slot lane is this lane's own)
        stx[lane] = stx[32 + lane];
        sti[lane] = sti[32 + lane];
      }
      queued = rest;
      __syncwarp();
      heavy(true, is, is, xs);
    }
  };
  auto drain = [&](auto&& heavy) {
    __syncwarp();
    const bool on = lane < queued;
    const int is = on ? sti[lane] : 0;
    heavy(on, is, is, on ? stx[lane] : 0.f);
    queued = 0;
  };

  // the request's cut: the tightest one its rows have published (one load);
  // while none is, and in every kCutScanEvery-th row, a snapshot of the
  // pool's bin counts (counts only grow, so a snapshot stays valid) and,
  // before the pool holds W candidates, the cut its seed gives, which the
  // row publishes
  if (tid == 0) sh.digit = (uint32_t)(kTailBins - 1) - __ldcg(&st->cutq);
  __syncthreads();
  int bcut = (int)sh.digit;
  __syncthreads();   // read before the scan below rewrites sh.digit
  if (bcut >= kTailBins - 1 || b % kCutScanEvery == 0) {
    block_scan_bins(gh, lh, (uint32_t)a.W, sh);
    int c = (int)sh.digit;
    if (seed != nullptr && c >= kTailBins - 1) {
      block_scan_bins(seed, lh, (uint32_t)a.W, sh);
      c = (int)sh.digit;
    }
    bcut = c < bcut ? c : bcut;
    if (tid == 0 && bcut < kTailBins - 1) atomicMax(&st->cutq, (uint32_t)(kTailBins - 1 - bcut));
  }
  // A logit below x_lo(bin) cannot reach that bin, and one at or above
  // x_hi(bin) reaches it or an earlier one: each bound lies one bin (1/64)
  // beyond the bin's edge, and near that edge the float32 roundings of the
  // score and of the bound move them by at most (|ref - cum| + |ref| + 128)
  // x 2^-23, under 1e-3 while |ref|, |cum| and |lse| stay below 4096 (log
  // probabilities always do; otherwise neither bound is used).  The Gumbel
  // noise has no bound, so kG keeps every candidate.
  const bool small = fabsf(ref) + fabsf(cum) + fabsf(lse) < 4096.f;
  auto x_lo = [&](int bin) -> float {
    return (kG || !small || bin >= kTailBins - 1) ? -INFINITY
                                                   : (ref - (float)(bin + 2) * (1.f / 64.f)) - cum + lse;
  };
  if (tid < kLadder) sh.warp_cnt[tid] = 0;
  for (int i = tid; i < kTailBins; i += kExpandThreads) lh[i] = 0;
  __syncthreads();
  // No request cut yet (fewer than W candidates in the pool): count, over the
  // first quarter of the row (at least 4 K candidates), the logits at or
  // above x_hi of each ladder bin B0 + ladder_bins(j); the lowest such bin
  // with K of them cuts the row (every candidate in a later bin ranks below
  // those K), so the passes below score only the candidates above it.  B0 is
  // the bin of the beam's own score, which no candidate exceeds by more than
  // rounding.
  if constexpr (!kG) {
    if (bcut >= kTailBins - 1 && n > kWideBuf && small) {
      const int b0 = score_bin(ref, cum);
      float th[kLadder];
      uint32_t c[kLadder];
#pragma unroll
      for (int j = 0; j < kLadder; ++j) {
        th[j] = (ref - (float)(b0 + ladder_bins(j)) * (1.f / 64.f)) - cum + lse;
        c[j] = 0;
      }
      auto count = [&](float x) {
#pragma unroll
        for (int j = 0; j < kLadder; ++j) c[j] += (x < th[j]) ? 0u : 1u;
      };
      if (vec) {
        const int nv = n >> 2;
        const int ns = min(nv, max(nv >> 2, K));   // float4 groups counted
        const float4* r4 = reinterpret_cast<const float4*>(row);
        for (int g0 = 0; g0 < ns; g0 += 4 * kExpandThreads) {
          float4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int g = g0 + u * kExpandThreads + tid;
            v[u] = g < ns ? __ldg(r4 + g) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            count(v[u].x);
            count(v[u].y);
            count(v[u].z);
            count(v[u].w);
          }
        }
      } else {
        const int ns = min(n, max(n >> 2, 4 * K));
        for (int i = tid; i < ns; i += kExpandThreads)
          count(__ldg(row + (code ? tb + __ldg(code + i) : i)));
      }
#pragma unroll
      for (int j = 0; j < kLadder; ++j) {
        const uint32_t t = __reduce_add_sync(0xffffffffu, c[j]);
        if (lane == 0) atomicAdd(&sh.warp_cnt[j], (int)t);
      }
      __syncthreads();
      for (int j = kLadder - 1; j >= 0; --j)   // the lowest ladder bin with K candidates
        if ((uint32_t)sh.warp_cnt[j] >= (uint32_t)K && b0 + ladder_bins(j) < bcut) bcut = b0 + ladder_bins(j);
    }
  }
  if (tid == 0) sh.cnt3 = 0;
  __syncthreads();
  // pass 1: histogram of the passing candidates' bins; the first kWideBuf
  // passing candidates are also kept, so that a row with few of them (every
  // row once the request's cut has formed) needs no second pass
  auto score1 = [&](bool on, int i, int tok, float x) {
    const uint32_t k = on ? cand_key<kG>(a, cum, lse, x, r, b, tok) : 0u;
    const int bin = on ? score_bin(ref, desc_key_value(k)) : kTailBins;
    const bool pass = on && bin <= bcut;
    if (pass) atomicAdd(lh + bin, 1u);
    const int pos = warp_reserve(&sh.cnt3, pass);
    if (pass && pos < kWideBuf) buf[pos] = ((unsigned long long)k << 32) | (uint32_t)i;
  };
  if constexpr (kG) {
    rounds(-INFINITY, score1);
  } else {
    rounds(x_lo(bcut), [&](bool keep, int i, int, float x) { stage(keep, i, x, score1); });
    drain(score1);
  }
  __syncthreads();
  {
    const int npass = sh.cnt3;
    if (npass <= kWideBuf) {   // every passing candidate is in the buffer
      const int take = npass < K ? npass : K;
      if (take == 0) return true;
      // the emitted candidates' bins: all of lh below bin D and take - below of bin D
      int D = kTailBins;
      uint32_t extra = 0;
      if (take < npass) {
        block_find_bin_smem(lh, (uint32_t)take, sh);
        D = (int)sh.digit;
        extra = (uint32_t)take - sh.below;
        smem_take_smallest(buf, npass, take, sh);
      }
      if (tid == 0) sh.pool_base = atomicAdd(&st->total, take);
      __syncthreads();
      const int base = sh.pool_base;
      for (int j = tid; j < take; j += kExpandThreads) {
        const unsigned long long e = buf[j];
        pool[base + j] = pool_key((uint32_t)(e >> 32), b, (int)(e & 0xFFFFFFFFull));
      }
      add_cut_hist(gh, lh, D, extra);
      return true;
    }
  }
  block_find_bin_smem(lh, (uint32_t)K, sh);
  const int D = (int)sh.digit;
  const uint32_t below = sh.below;
  const uint32_t nD = D < kTailBins ? lh[D] : 0u;
  __syncthreads();   // every thread has read the search's result before sh is reused
  if (nD > (uint32_t)kWideBuf) return false;
  const int take = D < kTailBins ? K : (int)below;
  const int need2 = D < kTailBins ? K - (int)below : 0;
  if (tid == 0) {
    sh.pool_base = take > 0 ? atomicAdd(&st->total, take) : 0;
    sh.cnt2 = 0;
    sh.cnt3 = 0;
  }
  __syncthreads();
  const int base = sh.pool_base;
  // pass 2: bins below D to the pool, bin D to the buffer
  const int blim = D < bcut ? D : bcut;
  auto score2 = [&](bool on, int i, int tok, float x) {
    const uint32_t k = on ? cand_key<kG>(a, cum, lse, x, r, b, tok) : 0u;
    const int bin = on ? score_bin(ref, desc_key_value(k)) : kTailBins;
    const bool pass = on && bin <= bcut;
    const bool direct = pass && bin < D;
    const bool atd = pass && bin == D;
    const int slot = warp_reserve(&sh.cnt2, direct);
    if (direct) pool[base + slot] = pool_key(k, b, i);
    const int pos = warp_reserve(&sh.cnt3, atd);
    if (atd) buf[pos] = ((unsigned long long)k << 32) | (uint32_t)i;   // pos < nD <= kWideBuf
  };
  if constexpr (kG) {
    rounds(-INFINITY, score2);
  } else {
    rounds(x_lo(blim), [&](bool keep, int i, int, float x) { stage(keep, i, x, score2); });
    drain(score2);
  }
  __syncthreads();
  if (need2 > 0) {
    const int first = sh.cnt2;   // == below
    __syncthreads();
    if (need2 < (int)nD) smem_take_smallest(buf, (int)nD, need2, sh);
    for (int j = tid; j < need2; j += kExpandThreads) {
      const unsigned long long e = buf[j];
      pool[base + first + j] = pool_key((uint32_t)(e >> 32), b, (int)(e & 0xFFFFFFFFull));
    }
  }
  add_cut_hist(gh, lh, D, need2 > 0 ? (uint32_t)need2 : 0u);
  return true;
}

// Fused a4 for one request, run by the last expand block of the request:
// select the min(W, pool) smallest pool keys, sort them, emit outputs.
template <bool kG>
__device__ void request_tail(const SelectArgs& a, ExpandShared& sh, const SelWs& ws, int r,
                             unsigned long long* keys) {
  const volatile SelState* st = ws.state + r;
  const int total = st->total;
  const int nt = total < a.W ? total : a.W;
  const unsigned long long* pool = ws.pool + (size_t)r * a.W * a.Kp;
  if (total == 0) {
    emit_outputs<kG>(a, ws, r, keys, 0);
    return;
  }
  // the request's score-bin histogram (complete: every block added its
  // candidates before taking its ticket), prefix-summed into shared memory
  // (the upper half of the key buffer); it brackets the nt-th best score
  uint32_t* hs = reinterpret_cast<uint32_t*>(keys + kTailCap / 2);
  // each live beam's first trie edge, for the output decode: its two dependent
  // loads are issued around the scan and the gather so their latency hides
  // behind them (one beam per thread; stored to sh.hist, free on the bucket path)
  const bool use_poff = a.has_trie && a.W <= kExpandThreads;
  const bool pf_live = use_poff && (int)threadIdx.x < a.n_live_in[r];
  int pnode = pf_live ? a.node_in[(size_t)r * a.W + threadIdx.x] : -1;
  block_scan_bins(ws.hist + (size_t)r * kBins, hs, (uint32_t)nt, sh);
  const int poffv = (pnode >= 0 && pnode < a.lvl.n_nodes) ? a.lvl.off[pnode] : 0;   // a bad node is never a parent
  const int Dbin = (int)sh.digit;
  const uint32_t c_le = sh.c_le;
  const float ref = bin_ref<kG>(a, a.cum_in[(size_t)r * a.W]);
  constexpr int kPer = 4;   // rounds of kPer x blockDim keys: the loads of a round overlap
  if (c_le <= (uint32_t)(2 * kExpandThreads)) {
    // bucket sort: the candidates of bins <= Dbin go to their bin's slots
    // (hs[b] = first slot of bin b, advanced as slots fill), then each one's
    // rank inside its bin settles its final place
    unsigned long long* tmp = keys;
    unsigned long long* sorted = keys + 2 * kExpandThreads;
    for (int c0 = 0; c0 < total; c0 += kPer * kExpandThreads) {
      unsigned long long kv[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = c0 + u * kExpandThreads + threadIdx.x;
        kv[u] = i < total ? __ldcg(pool + i) : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = c0 + u * kExpandThreads + threadIdx.x;
        const int bin = score_bin(ref, desc_key_value((uint32_t)(kv[u] >> 32)));
        const bool on = i < total && bin <= Dbin;
        const uint32_t slot = warp_bin_reserve(hs, (uint32_t)bin, on);
        if (on && slot < c_le) tmp[slot] = kv[u];
      }
    }
    if (pf_live) sh.hist[threadIdx.x] = (uint32_t)poffv;
    __syncthreads();
    // after the fill hs[b] is the end of bin b and hs[b - 1] its start
    for (int j = threadIdx.x; j < (int)c_le; j += kExpandThreads) {
      const unsigned long long k = tmp[j];
      const int bin = score_bin(ref, desc_key_value((uint32_t)(k >> 32)));
      const uint32_t end = min(hs[bin], c_le);
      const uint32_t start = bin > 0 ? min(hs[bin - 1], end) : 0u;
      uint32_t rank = start;
      for (uint32_t m = start; m < end; ++m) rank += tmp[m] < k ? 1u : 0u;
      if (rank < (uint32_t)nt) sorted[rank] = k;
    }
    __syncthreads();
    emit_outputs<kG>(a, ws, r, sorted, nt, use_poff ? reinterpret_cast<const int*>(sh.hist) : nullptr);
    return;
  }
  int nc = 0;
  if (c_le <= (uint32_t)kTailCap) {
    if (threadIdx.x == 0) sh.count = 0;
    __syncthreads();
    for (int c0 = 0; c0 < total; c0 += kPer * kExpandThreads) {
      unsigned long long kv[kPer];
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int i = c0 + u * kExpandThreads + threadIdx.x;
        kv[u] = i < total ? __ldcg(pool + i) : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {   // the sort below orders them: slots are unordered
        const int i = c0 + u * kExpandThreads + threadIdx.x;
        const bool flag =
            (i < total) && score_bin(ref, desc_key_value((uint32_t)(kv[u] >> 32))) <= Dbin;
        const int pos = warp_reserve(&sh.count, flag);
        if (flag && pos < kTailCap) keys[pos] = kv[u];
      }
    }
    __syncthreads();
    nc = sh.count < kTailCap ? sh.count : kTailCap;
    goto selected;
  }
  {   // many candidates at about the same score: radix narrowing over the pool
    unsigned long long prefix = 0;
    int shift = 64;
    uint32_t need = (uint32_t)nt, sure = 0, in_bin = 0;
    while (true) {
      in_bin = narrow_pass<true>(pool, total, prefix, shift, need, sure, sh);
      if (sure + in_bin <= (uint32_t)kTailCap || shift == 0) break;
    }
    if (threadIdx.x == 0) sh.count = 0;
    __syncthreads();
    for (int c0 = 0; c0 < total; c0 += blockDim.x) {   // block-uniform trip count
      const int i = c0 + threadIdx.x;
      const unsigned long long k = i < total ? __ldcg(pool + i) : 0ull;
      const bool flag = i < total && (k >> shift) <= prefix;
      const int pos = warp_reserve(&sh.count, flag);
      if (flag && pos < kTailCap) keys[pos] = k;
    }
    __syncthreads();
    nc = sh.count < kTailCap ? sh.count : kTailCap;
  }
selected:
  __syncthreads();
  if (nc <= 2 * kExpandThreads) {   // small candidate sets: sort them all, keep the first nt
    block_sort_small(keys, nc);
    emit_outputs<kG>(a, ws, r, keys, nt);
    return;
  }
  if (nc > nt) {   // exact threshold: narrow until the keys at or below it number nt
    unsigned long long prefix = 0;
    int shift = 64;
    uint32_t need = (uint32_t)nt, sure = 0;
    while (true) {
      const uint32_t in_bin = narrow_pass<false>(keys, nc, prefix, shift, need, sure, sh);
      if (sure + in_bin == (uint32_t)nt || shift == 0) break;
    }
    // in-place compaction of the winners to keys[0..nt)
    if (threadIdx.x == 0) sh.count = 0;
    __syncthreads();
    for (int c0 = 0; c0 < nc; c0 += blockDim.x) {
      const int i = c0 + threadIdx.x;
      unsigned long long k = 0;
      int flag = 0;
      if (i < nc) {
        k = keys[i];
        flag = (k >> shift) <= prefix;
      }
      int tot;
      const int rk = block_rank(flag, sh.warp_cnt, &tot);   // all reads of the chunk precede writes
      if (flag) keys[sh.count + rk] = k;
      __syncthreads();
      if (threadIdx.x == 0) sh.count += tot;
      __syncthreads();
    }
  }
  if (nt <= 2 * kExpandThreads) {   // winners now in keys[0..nt)
    block_sort_small(keys, nt);
    emit_outputs<kG>(a, ws, r, keys, nt);
    return;
  }
  int np = 32;
  while (np < nt) np <<= 1;
  for (int i = nt + threadIdx.x; i < np; i += blockDim.x) keys[i] = ~0ull;
  __syncthreads();
  bitonic_sort(keys, np);
  emit_outputs<kG>(a, ws, r, keys, nt);
}

// a2-a5 for live beam b of request r once its log-sum-exp is known: the
// row's candidates go to the request's pool; with kFused the last row of the
// request to finish (a per-request ticket) runs the request's global top-W.
// Dynamic shared memory: the row's key cache (32 KB); the fused tail reuses it
// for candidate keys after the ticket.
template <bool kFused, bool kPf, bool kG, bool kD>
__device__ __forceinline__ void expand_and_select(const SelectArgs& a, ExpandShared& sh, const SelWs& ws,
                                                  int r, int b, int nl, float lse,
                                                  unsigned char* tail_smem) {
  const int tid = threadIdx.x;
  uint32_t* kcache = reinterpret_cast<uint32_t*>(tail_smem);
  expand_candidates<kPf, kG, kD>(a, sh, ws, r, b, (kFused ? ws.hist : ws.cuthist) + (size_t)r * kBins,
                                 kcache, lse);
  if constexpr (kFused) {
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      sh.count = atomicAdd(&ws.state[r].tickets, 1);
    }
    __syncthreads();
    if (sh.count != nl - 1) return;
    __threadfence();
    request_tail<kG>(a, sh, ws, r, reinterpret_cast<unsigned long long*>(tail_smem));
  }
}

// a2-a5 when the caller supplies the row normalisers (lse_in): one block per
// live beam.  The deterministic variants fit 64 registers, two blocks per SM.
template <bool kFused, bool kG, bool kD>
__global__ void __launch_bounds__(kExpandThreads, kG ? 1 : 2)
bd_expand_kernel(SelectArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // as in the stream kernel
  __shared__ ExpandShared sh;
  extern __shared__ __align__(16) unsigned char tail_smem[];
  const int r = blockIdx.x, b = blockIdx.y;   // the first rows of every request run first
  SelWs ws = carve(a.ws, a.R, a.W, a.Kp);
  if (b == 0 && r == 0 && threadIdx.x == 0) ws.hdr->bar_count = 0u;
  const int nl = a.n_live_in[r];
  if (b >= nl) return;
  const float lse = a.lse_in[(size_t)r * a.W + b];
  expand_and_select<kFused, false, kG, kD>(a, sh, ws, r, b, nl, lse, tail_smem);
}

// Seeds of the open-vocabulary requests' cuts, before their rows expand (the
// rows that start while a request's pool holds fewer than W candidates
// would otherwise have no cut).  Every thread takes the maximum of `span`
// consecutive logits of one of a request's first kSeedRows live rows and
// counts the score bin the expansion computes for that candidate in the
// request's seed histogram.  Each maximum is a real candidate of its row,
// and span >= V / K keeps a row's maxima at most K, so a row holding x of
// them at or above a bin holds at least x of its top_k there: once W of them
// lie at or above bin b*, a candidate in a later bin ranks below W pool
// candidates, which is the request's cut.
constexpr int kSeedRows = 16;
inline int seed_span(int V, int K) {
  int s = (V + K - 1) / K;
  if (s < 16) s = 16;
  return (s + 3) & ~3;   // whole float4 groups
}
__global__ void __launch_bounds__(kExpandThreads) bd_seed_kernel(SelectArgs a, int span) {
  __shared__ uint32_t bins[kTailBins];   // the block's counts, added to the request's once per bin
  const int r = blockIdx.z, b = blockIdx.y;
  if (b >= a.n_live_in[r]) return;
  for (int i = threadIdx.x; i < kTailBins; i += kExpandThreads) bins[i] = 0;
  const SelWs ws = carve(a.ws, a.R, a.W, a.Kp);
  const size_t rowi = (size_t)r * a.W + b;
  const float* row = a.logits + rowi * (size_t)a.row_stride;
  const long long i0 = ((long long)blockIdx.x * kExpandThreads + threadIdx.x) * span;
  const bool on = i0 < a.V;
  float m = -INFINITY;
  if (on) {
    const int n = (int)min((long long)span, (long long)a.V - i0);
    const float* x = row + i0;
    int j = 0;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
      const float4* x4 = reinterpret_cast<const float4*>(x);
#pragma unroll 8
      for (; j + 4 <= n; j += 4) {
        const float4 v = __ldg(x4 + (j >> 2));
        m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
      }
    }
    for (; j < n; ++j) m = fmaxf(m, __ldg(x + j));
  }
  const float lse = a.lse_in[rowi];   // the caller's, or the normaliser stream's in the workspace
  const float cum = a.cum_in[rowi];
  const float ref = bin_ref<false>(a, a.cum_in[(size_t)r * a.W]);
  const uint32_t k = on ? cand_key<false>(a, cum, lse, m, r, b, 0) : 0u;
  __syncthreads();   // the block's bins are zero
  if (on) atomicAdd(bins + score_bin(ref, desc_key_value(k)), 1u);
  __syncthreads();
  uint32_t* sh = ws.seedhist + (size_t)r * kBins;
  for (int i = threadIdx.x; i < kTailBins; i += kExpandThreads)
    if (bins[i] != 0u) atomicAdd(sh + i, bins[i]);
}

// The whole selection step in one launch: S blocks per live logits row each
// fold (max, sum of exp) of one chunk of the row (a1); the last of them (a
// per-row ticket) combines the chunks into the row's log-sum-exp and goes on
// with the row (a2, a3) while the row is still in L2; with kFused the last
// row of each request selects the request's top-W (a4, a5).  The stream
// part holds nothing else, so the kernel fits 32 registers and four
// 512-thread blocks per SM keep enough loads in flight.
template <bool kFused, bool kG>
__global__ void __launch_bounds__(kExpandThreads, 4)
bd_stream_select_kernel(SelectArgs a) {
  // a kernel launched after this one with programmatic stream serialization
  // may start once every block of this grid has begun; it must wait for the
  // grid's completion before reading any of its outputs
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  __shared__ ExpandShared sh;
  extern __shared__ __align__(16) unsigned char tail_smem[];
  const int S = a.row_splits;
  const int b = blockIdx.x / S, sidx = blockIdx.x - b * S, r = blockIdx.y, tid = threadIdx.x;
  SelWs ws = carve(a.ws, a.R, a.W, a.Kp);
  if (blockIdx.x == 0 && r == 0 && tid == 0) ws.hdr->bar_count = 0u;
  const int nl = a.n_live_in[r];
  if (b >= nl) return;
  const size_t rowi = (size_t)r * a.W + b;
  const float* row = a.logits + rowi * (size_t)a.row_stride;
  const int c0 = sidx * a.row_chunk;
  const int c1 = min(a.V, c0 + a.row_chunk);
  const float2 ms = stream_max_sum(row, c0, c1, sh);
  // the row's expansion inputs, fetched by another warp while thread 0
  // publishes the chunk and takes the row ticket (a block that turns out not
  // to be the row's last just drops them)
  if (tid == 32) {
    sh.pf_cum = a.cum_in[rowi];
    sh.pf_ref = a.cum_in[(size_t)r * a.W];
    int e0 = 0, e1 = a.V;
    if (a.has_trie) {
      const int node = a.node_in[rowi];
      const bool bad = node < 0 || node >= a.lvl.n_nodes;
      e0 = bad ? -2 : a.lvl.off[node];
      e1 = bad ? -2 : a.lvl.off[node + 1];
    }
    sh.pf_e0 = e0;
    sh.pf_e1 = e1;
  }
  float lse;
  if (S == 1) {
    __syncthreads();
    lse = ms.x + logf(ms.y);
  } else {
    if (tid == 0) {
      ws.rowpart[rowi * kMaxRowSplits + sidx] = ms;
      __threadfence();
      sh.count = atomicAdd(ws.rowtick + rowi, 1);
    }
    __syncthreads();
    if (sh.count != S - 1) return;
    __threadfence();
    if (tid < 32) {   // one warp: lane k holds chunk k's (max, sum)
      const float2 p = tid < S ? __ldcg(ws.rowpart + rowi * kMaxRowSplits + tid)
                               : make_float2(-INFINITY, 0.f);
      float M = p.x;
      for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      float tot = (p.y > 0.f) ? p.y * ex2((p.x - M) * kLog2e) : 0.f;
      for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
      if (tid == 0) sh.lse = M + logf(tot);
    }
    __syncthreads();
    lse = sh.lse;
  }
  if (tid == 0 && a.lse_out != nullptr) a.lse_out[rowi] = lse;
  // the candidates are scored against the caller's normaliser when one is
  // given (the rest of the launch is the same code path)
  if (a.score_lse != nullptr) lse = __ldg(a.score_lse + rowi);
  // the outputs' score recomputation (Gumbel) and the expansion kernel
  // (lse-only mode) read the scoring normaliser back
  if ((kG || a.lse_only) && tid == 0) ws.rowlse[rowi] = lse;
  if (a.lse_only) return;
  expand_and_select<kFused, true, kG, false>(a, sh, ws, r, b, nl, lse, tail_smem);
}

// ---------------------------------------------------------------------------
struct GlobalSmem {
  uint32_t hist[kBins];
  int warp_cnt[32];
  uint32_t digit, below;
  int all_done;
};

constexpr size_t kGlobalKeysOffset = (sizeof(GlobalSmem) + 15) & ~(size_t)15;

__global__ void __launch_bounds__(kGlobalThreads)
bd_global_kernel(SelectArgs a) {
  extern __shared__ __align__(16) unsigned char dyn[];
  GlobalSmem& sh = *reinterpret_cast<GlobalSmem*>(dyn);
  unsigned long long* keys = reinterpret_cast<unsigned long long*>(dyn + kGlobalKeysOffset);
  const int tid = threadIdx.x;
  const unsigned G = gridDim.x;
  SelWs ws = carve(a.ws, a.R, a.W, a.Kp);

  // phase 0: targets.  Small pools skip straight to the sort.  The expansion
  // counted every pool key in the request's score-bin histogram (cuthist);
  // when the bin holding the nt-th best key closes a prefix of at most
  // kSelectCap keys, the pool is gathered by bin and the radix passes are
  // skipped.
  for (int r = blockIdx.x; r < a.R; r += G) {
    volatile SelState* st = ws.state + r;
    const int total = st->total;
    const int nt = total < a.W ? total : a.W;
    const bool big = total > kSelectCap && nt > 0;   // block-uniform
    if (big) {
      const uint32_t* ch = ws.cuthist + (size_t)r * kBins;
      for (int i = tid; i < kBins; i += kGlobalThreads) sh.hist[i] = __ldcg(ch + i);
      if (tid == 0) sh.digit = kBins;   // stays kBins if the bins hold fewer than nt keys
      __syncthreads();
      if (tid < 32) warp_find_digit(sh.hist, kBins, (uint32_t)nt, &sh.digit, &sh.below);
      __syncthreads();
    }
    if (tid == 0) {
      const bool by_bin = big && sh.digit < (uint32_t)kBins && sh.below + sh.hist[sh.digit] <= (uint32_t)kSelectCap;
      st->n_target = nt;
      st->need = nt;
      st->sure = 0;
      st->prefix = 0ull;
      st->shift = 64;
      st->ncand = 0;
      st->bin_mode = by_bin ? 1 : 0;
      st->bin_cut = by_bin ? (int)sh.digit : 0;
      st->done = (total <= kSelectCap || by_bin) ? 1 : 0;
    }
    __syncthreads();   // sh is reused for the next request
  }
  grid_barrier(ws.hdr, G);

  // radix-select passes over 12-bit digits until every request has at most
  // kSelectCap keys at or below its threshold prefix
  for (int pass = 0; pass < 6; ++pass) {
    if (tid == 0) {
      int all = 1;
      for (int r = 0; r < a.R; ++r) all &= ((volatile SelState*)(ws.state + r))->done;
      sh.all_done = all;
    }
    __syncthreads();
    if (sh.all_done) break;
    const int width = pass < 5 ? kDigitBits : 4;
    for (int r = 0; r < a.R; ++r) {
      volatile SelState* st = ws.state + r;
      if (st->done) continue;
      const int shift = st->shift;
      const unsigned long long prefix = st->prefix;
      const int nshift = shift - width;
      const int total = st->total;
      for (int i = tid; i < (1 << width); i += kGlobalThreads) sh.hist[i] = 0;
      __syncthreads();
      const unsigned long long* pool = ws.pool + (size_t)r * a.W * a.Kp;
      const int per = (total + G - 1) / G;
      const int i0 = blockIdx.x * per, i1 = min(total, i0 + per);
      for (int i = i0 + tid; i < i1; i += kGlobalThreads) {
        const unsigned long long k = pool[i];
        if (shift == 64 || (k >> shift) == prefix)
          atomicAdd(&sh.hist[(uint32_t)(k >> nshift) & ((1u << width) - 1u)], 1u);
      }
      __syncthreads();
      uint32_t* gh = ws.hist + (size_t)r * kBins;
      for (int i = tid; i < (1 << width); i += kGlobalThreads)
        if (sh.hist[i]) atomicAdd(gh + i, sh.hist[i]);
      __syncthreads();
    }
    grid_barrier(ws.hdr, G);
    for (int r = blockIdx.x; r < a.R; r += G) {
      volatile SelState* st = ws.state + r;
      if (st->done) continue;
      volatile uint32_t* gh = ws.hist + (size_t)r * kBins;
      for (int i = tid; i < (1 << width); i += kGlobalThreads) sh.hist[i] = gh[i];   // to shared memory
      __syncthreads();
      if (tid < 32) warp_find_digit(sh.hist, 1 << width, (uint32_t)st->need, &sh.digit, &sh.below);
      __syncthreads();
      if (tid == 0) {
        const uint32_t D = sh.digit;
        const uint32_t in_bin = sh.hist[D];
        st->sure += (int)sh.below;
        st->need -= (int)sh.below;
        st->prefix = (st->prefix << width) | D;
        st->shift -= width;
        if (st->sure + (int)in_bin <= kSelectCap || st->shift == 0) st->done = 1;
      }
      __syncthreads();
      for (int i = tid; i < (1 << width); i += kGlobalThreads) gh[i] = 0;
      __syncthreads();
    }
    grid_barrier(ws.hdr, G);
  }

  // gather every key at or below the threshold prefix (bin mode: in a score
  // bin up to the cut, the bin computed as the expansion computed it)
  for (int r = 0; r < a.R; ++r) {
    volatile SelState* st = ws.state + r;
    const int shift = st->shift;
    const unsigned long long prefix = st->prefix;
    const int total = st->total;
    const bool by_bin = st->bin_mode != 0;
    const int bin_cut = st->bin_cut;
    const float cum0 = a.cum_in[(size_t)r * a.W];
    const float ref = a.inv_tau > 0.f ? bin_ref<true>(a, cum0) : bin_ref<false>(a, cum0);
    const unsigned long long* pool = ws.pool + (size_t)r * a.W * a.Kp;
    unsigned long long* cand = ws.cand + (size_t)r * kSelectCap;
    const int per = (total + G - 1) / G;
    const int i0 = blockIdx.x * per, i1 = min(total, i0 + per);
    for (int c0 = i0; c0 < i1; c0 += kGlobalThreads) {
      const int i = c0 + tid;
      unsigned long long k = 0;
      int flag = 0;
      if (i < i1) {
        k = pool[i];
        flag = by_bin ? score_bin(ref, desc_key_value((uint32_t)(k >> 32))) <= bin_cut
                      : (shift == 64) || ((k >> shift) <= prefix);
      }
      int tot;
      const int rk = block_rank(flag, sh.warp_cnt, &tot);
      if (tid == 0 && tot) sh.below = (uint32_t)atomicAdd((int*)&st->ncand, tot);
      __syncthreads();
      const int pos = (int)sh.below + rk;
      if (flag) {
        if (pos < kSelectCap) cand[pos] = k;
        else set_status(ws.hdr, BEAMDEC_ERR_DEVICE_CHECK);
      }
      __syncthreads();
    }
  }
  grid_barrier(ws.hdr, G);

  // per request: the survivors' keys are distinct, so each one's rank among
  // them (a count of smaller keys) is its output row.  The request's slices
  // of kRankSlice survivors are dealt round the grid; a block holds all of
  // the request's survivors in shared memory and eight threads rank each key.
  constexpr int kRankSlice = kGlobalThreads / 8;
  int wbase = 0;   // slices of the requests before r (the same in every block)
  for (int r = 0; r < a.R; ++r) {
    const volatile SelState* st = ws.state + r;
    const int nc = min((int)st->ncand, kSelectCap);
    const int nt = st->n_target;
    const int ns = (nc + kRankSlice - 1) / kRankSlice;
    const unsigned long long* cand = ws.cand + (size_t)r * kSelectCap;
    const int first = (int)((blockIdx.x + G - (unsigned)(wbase % (int)G)) % G);
    wbase += ns;
    if (first >= ns) continue;   // block-uniform
    for (int i = tid; i < nc; i += kGlobalThreads) keys[i] = __ldcg(cand + i);
    __syncthreads();
    const int part = tid & 7;
    for (int sl = first; sl < ns; sl += G) {
      const int q = sl * kRankSlice + (tid >> 3);
      const unsigned long long kq = q < nc ? keys[q] : 0ull;
      int rank = 0;
      for (int i = part; i < nc; i += 8) rank += keys[i] < kq ? 1 : 0;
      rank += __shfl_xor_sync(0xffffffffu, rank, 1);
      rank += __shfl_xor_sync(0xffffffffu, rank, 2);
      rank += __shfl_xor_sync(0xffffffffu, rank, 4);
      if (q < nc && rank < nt) {
        if (a.inv_tau > 0.f) emit_row<true>(a, ws, r, rank, kq, part);
        else emit_row<false>(a, ws, r, rank, kq, part);
      }
    }
    __syncthreads();   // every rank is counted before the next request's keys arrive
  }
  // rows past each request's n_target, and n_live_out
  const size_t nrows = (size_t)a.R * a.W;
  for (size_t e = (size_t)blockIdx.x * kGlobalThreads + tid; e < nrows; e += (size_t)G * kGlobalThreads) {
    const int r = (int)(e / a.W), j = (int)(e - (size_t)r * a.W);
    const int nt = ((const volatile SelState*)(ws.state + r))->n_target;
    if (j >= nt) emit_dead_row(a, r, j);
    if (j == 0) a.n_live_out[r] = nt;
  }
}

struct GlobalLaunchCfg {
  int max_blocks = 0;
  size_t smem = 0;
};

}  // namespace

template <bool kG, bool kD>
void launch_expand(bool fused, dim3 grid, size_t dsm, cudaStream_t stream, const SelectArgs& a) {
  if (fused) bd_expand_kernel<true, kG, kD><<<grid, kExpandThreads, dsm, stream>>>(a);
  else bd_expand_kernel<false, kG, kD><<<grid, kExpandThreads, dsm, stream>>>(a);
}

size_t select_workspace_bytes(int R, int W, int K, int V) {
  const int Kp = K < V ? K : V;
  return kWsHeaderBytes + align256((size_t)R * sizeof(SelState)) +
         align256((size_t)R * W * sizeof(int32_t)) +
         3 * align256((size_t)R * kBins * sizeof(uint32_t)) + align256((size_t)R * W * Kp * 8) +
         align256((size_t)R * kSelectCap * 8) +
         align256((size_t)R * W * kMaxRowSplits * sizeof(float2)) + (size_t)R * W * sizeof(float);
}

int launch_select(const SelectArgs& a, cudaStream_t stream) {
  static GlobalLaunchCfg cfg[64];
  static PerDeviceOnce cfg_once;
  const size_t smem = kGlobalKeysOffset + (size_t)kSelectCap * 8;
  const int crc = once_per_device(cfg_once, [smem](int d) {
    if (cudaFuncSetAttribute(bd_global_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return BEAMDEC_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bd_global_kernel, kGlobalThreads,
                                                      smem) != cudaSuccess || per_sm < 1)
      return BEAMDEC_ERR_CUDA;
    cfg[d].max_blocks = per_sm * sm_count();
    cfg[d].smem = smem;
    // two expansion blocks per SM need more shared memory than the driver's
    // default split gives one kernel
    const void* row_kernels[] = {
        (const void*)bd_expand_kernel<false, false, false>, (const void*)bd_expand_kernel<false, false, true>,
        (const void*)bd_expand_kernel<false, true, false>,  (const void*)bd_expand_kernel<false, true, true>,
        (const void*)bd_expand_kernel<true, false, false>,  (const void*)bd_expand_kernel<true, false, true>,
        (const void*)bd_expand_kernel<true, true, false>,   (const void*)bd_expand_kernel<true, true, true>};
    for (const void* f : row_kernels)
      if (cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return BEAMDEC_ERR_CUDA;
    return BEAMDEC_OK;
  });
  if (crc != BEAMDEC_OK) return crc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BEAMDEC_ERR_CUDA;
  SelectArgs a2 = a;
  // blocks per logits row: about 25K logits each (the row's tail of partial
  // waves shrinks with the work unit), at most kMaxRowSplits.  At V = 151936
  // and 2048 rows, 6 blocks per row measured 204 us against 206 us for 4 and
  // 215 us for 5, 7 or 8.
  int S = a.V / 25000;
  if (S < 1) S = 1;
  if (S > kMaxRowSplits) S = kMaxRowSplits;
  int chunk = ((a.V + S - 1) / S + 3) & ~3;
  S = (a.V + chunk - 1) / chunk;
  a2.row_splits = S;
  a2.row_chunk = chunk;
  SelWs ws = carve(a.ws, a.R, a.W, a.Kp);
  const size_t zero_bytes = (char*)ws.pool - (char*)ws.state;
  if (cudaMemsetAsync(ws.state, 0, zero_bytes, stream) != cudaSuccess) return BEAMDEC_ERR_CUDA;

  // Pools of at most 1M keys per request (W <= 4096) are selected by the last
  // row of each request inside the launch; larger ones by the cooperative
  // grid kernel afterwards.
  const bool fused = a.W <= kTailCap && (long long)a.W * a.Kp <= (1ll << 20);
  static_assert(kKeyCache * 4 <= kTailCap * 8, "fused dynamic shared memory");
  const size_t dsm = fused ? kTailCap * sizeof(unsigned long long) : kKeyCache * sizeof(uint32_t);
  const bool gumbel = a.inv_tau > 0.f;
  const bool dense = a.has_trie && a.lvl.mask != nullptr;
  // Open-vocabulary rows wider than the key cache, and levels with dense
  // child masks: the one-launch kernel only streams each row for its
  // normaliser (kept in the workspace), and the expansion kernel, whose
  // register budget holds the wide-row select and the mask enumeration,
  // expands the rows.
  const bool two_phase =
      a.lse_in == nullptr && (dense || (!a.has_trie && a.V > kKeyCache && a.K < a.V));
  if (two_phase) {
    SelectArgs s1 = a2;
    s1.lse_only = 1;
    dim3 g0(a.W * S, a.R);
    prof_begin(kKStream, stream);
    if (gumbel) bd_stream_select_kernel<false, true><<<g0, kExpandThreads, dsm, stream>>>(s1);
    else bd_stream_select_kernel<false, false><<<g0, kExpandThreads, dsm, stream>>>(s1);
    prof_end(kKStream, stream);
    if (cudaGetLastError() != cudaSuccess) return BEAMDEC_ERR_CUDA;
    a2.lse_in = ws.rowlse;   // the scoring normaliser of every live row
    a2.lse_out = nullptr;    // already written with the kernel's own value
    a2.score_lse = nullptr;
  }
  if (a2.lse_in != nullptr && !gumbel && !a.has_trie && a.V > kKeyCache && a.K < a.V) {
    // seeds of the requests' cuts for the open-vocabulary expansion
    const int span = seed_span(a.V, a.K);
    const int per_block = kExpandThreads * span;
    const dim3 gs((unsigned)((a.V + per_block - 1) / per_block), kSeedRows, (unsigned)a.R);
    prof_begin(kKSeed, stream);
    bd_seed_kernel<<<gs, kExpandThreads, 0, stream>>>(a2, span);
    prof_end(kKSeed, stream);
    if (cudaGetLastError() != cudaSuccess) return BEAMDEC_ERR_CUDA;
    a2.seeded = 1;
  }
  if (a2.lse_in == nullptr) {
    dim3 g0(a.W * S, a.R);
    prof_begin(kKStream, stream);
    if (gumbel) {
      if (fused) bd_stream_select_kernel<true, true><<<g0, kExpandThreads, dsm, stream>>>(a2);
      else bd_stream_select_kernel<false, true><<<g0, kExpandThreads, dsm, stream>>>(a2);
    } else {
      if (fused) bd_stream_select_kernel<true, false><<<g0, kExpandThreads, dsm, stream>>>(a2);
      else bd_stream_select_kernel<false, false><<<g0, kExpandThreads, dsm, stream>>>(a2);
    }
    prof_end(kKStream, stream);
  } else {
    // requests inner: until W candidates of a request reach its pool, its
    // rows meet no cut and cost an extra pass, so the first rows of all
    // requests share the first wave of blocks
    const dim3 g1(a.R, a.W);
    prof_begin(kKExpand, stream);
    if (gumbel) {
      if (dense) launch_expand<true, true>(fused, g1, dsm, stream, a2);
      else launch_expand<true, false>(fused, g1, dsm, stream, a2);
    } else {
      if (dense) launch_expand<false, true>(fused, g1, dsm, stream, a2);
      else launch_expand<false, false>(fused, g1, dsm, stream, a2);
    }
    prof_end(kKExpand, stream);
  }
  if (cudaGetLastError() != cudaSuccess) return BEAMDEC_ERR_CUDA;
  if (fused) return BEAMDEC_OK;

  const long long pool_max = (long long)a.R * a.W * a.Kp;
  long long want = (pool_max + 4095) / 4096;
  if (want < a.R) want = a.R;
  int grid = (int)(want < cfg[dev].max_blocks ? want : cfg[dev].max_blocks);
  if (grid < 1) grid = 1;
  SelectArgs copy = a2;
  void* params[] = {&copy};
  prof_begin(kKGlobal, stream);
  const cudaError_t e = cudaLaunchCooperativeKernel((const void*)bd_global_kernel, dim3(grid),
                                                    dim3(kGlobalThreads), params, cfg[dev].smem,
                                                    stream);
  prof_end(kKGlobal, stream);
  return e == cudaSuccess ? BEAMDEC_OK : BEAMDEC_ERR_CUDA;
}

}  // namespace bd
