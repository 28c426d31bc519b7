// Shared stage of the beam attention on the tcgen05 tensor cores.
//
// "Generative recommendation design" (xLLM) §4.2.1-§4.2.2: the prompt KV of a
// request is stored once and all of its beams attend to it, so for one
// (request, kv head g) the queries of every beam and every query head of the
// group form one dense matrix Q [W*G x d] against the prompt's K and V: the
// shared stage is a flash-attention contraction with M = W*G rows.  Its
// output is the partial (max, sum, unnormalised output) of every query row,
// merged later with the unshared stage (§4.2.2).  When the whole prompt is
// one split, every row's shared partial stays in its CTA, so the epilogue
// runs the unshared stage and the merge itself and writes the output rows;
// otherwise the partials go to the merge kernel.
//
// One CTA owns 256 query rows (two 128-row tiles) of one (request, kv head,
// prompt split), so every K/V tile it loads feeds two tiles of MMAs:
//   warp 8       TMA producer: Q once, then K and V tiles of 128 keys (two
//                64-column SWIZZLE_128B boxes each) through a 5-slot ring
//                (two and a half chunks ahead of the MMAs);
//   warp 9       allocates TMEM and issues every MMA from one thread, in the
//                order S0(c) S1(c) | PV0(c) S0(c+1) | PV1(c) S1(c+1) | ... so
//                the tensor core works on one tile while the other tile's
//                softmax runs;
//   warps 0-3    softmax of tile 0, warps 4-7 softmax of tile 1: thread t
//                owns row t (TMEM lane t); reads its 128 scores from TMEM
//                twice (row max, then P; one 128-column load each), keeps
//                max/sum in log2 units and writes P (bf16, two per column)
//                back into TMEM over the first 64 columns of its S tile,
//                where the PV MMA reads it as its A operand.
//   warp 10      when the merge is fused (one prompt split): pulls the CTA's
//                unshared K/V rows into L2 for the epilogue.
// The output O accumulates in TMEM across chunks (S0 O0 S1 O1, 128 columns
// each).  P_t(c) overwrites S_t(c) only after the softmax has read all of it,
// and S_t(c+1) is issued after PV_t(c) by the same thread, so the tensor core
// reads P before the next S lands on it.  The running max used for P only moves when a chunk's max exceeds
// it by more than 2^8; then the warp rescales its O rows in TMEM before the
// next PV.  That keeps P <= 2^8 and leaves the result exact.  The commit that
// signals S_t(c+1) also covers PV_t(c) (a commit tracks every earlier MMA of
// the issuing thread), so the softmax of chunk c+1 may overwrite P_t and
// touch O_t once it has seen S_t(c+1).  Keeping P out of shared memory frees
// the ring's extra slots and the shared-memory bandwidth P would take.
// Every mbarrier wait is bounded; a timeout records BEAMDEC_ERR_TIMEOUT, ends
// the loops and still frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>

#include <utility>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace bd {
namespace {

using namespace tc;

constexpr int kThreads = 352;   // warps 0-7 softmax, 8 TMA, 9 MMA, 10 L2 prefetch
constexpr uint32_t kHalfBytes = 16384;           // 128 rows x 128 B
constexpr uint32_t kTileBytes = 2 * kHalfBytes;  // 128 x 128 bf16
constexpr int kSlots = 5;                        // K/V ring
constexpr uint32_t kOffQ = 0;                    // Q0, Q1
constexpr uint32_t kOffKV = 2 * kTileBytes;      // kSlots tiles
constexpr uint32_t kSmemBytes = kOffKV + kSlots * kTileBytes + 1024;
constexpr uint32_t kTmemCols = 512;              // S0 O0 S1 O1
constexpr float kRescale = 8.f;                  // log2 headroom before O is rescaled
// unshared tokens the fused epilogue takes (its scratch, a score and a slot
// per token for each of a tile's 128 rows in the tile's 64 KB of the idle
// ring, holds 64).  One thread per row walks its tokens one at a time, so
// each token costs every CTA a few dependent memory round trips, while the
// merge kernel (a warp per beam and kv head, four tokens in flight) pays the
// partials' round trip through memory once.  Measured on 2 x 5000 beams, 16
// query and 8 kv heads, a 1024-key prompt: fused 136 us + 39 us per token
// after the first, against 271 us + 14.6 us per token with the merge kernel.
constexpr int kFusedMaxL = 6;

// MN-major B operand (V, d contiguous): the leading byte offset is the stride
// between the two 64-column swizzle atoms along d (the two 16 KB halves), the
// stride byte offset the stride between groups of 8 keys (8 x 128 B).
constexpr uint32_t kVLbo = kHalfBytes;
constexpr uint32_t kVSbo = 1024;

struct TcParams {
  int R, W, Hq, Hkv, G, rows, split_len;
  // launched as a programmatic dependent of the previous kernel: wait for it
  // before reading the slot table or the live counts (late: after the main
  // loop; early: before everything, so dead tiles can skip the main loop)
  int dep_wait_late;
  // e4m3 KV prepared earlier: the workspace's record of the prompt K/V its
  // bf16 copy came from must name these (else BEAMDEC_ERR_DEVICE_CHECK)
  const void* prep_k;
  const void* prep_v;
  const void* prep_dst;   // where this call's maps read the copy
  float scale_log2;   // sm_scale * log2(e)
  const float* k_scale;   // per kv head; fp8 KV only (nullptr otherwise)
  int64_t shared_rows;
  const int32_t* prompt_offsets;
  const int32_t* n_live;
  float* pm;
  float* pl;
  float* po;
  WsHeader* hdr;
  // fuse != 0: the prompt is one split, so the epilogue runs the unshared
  // stage and the merge itself and writes the output rows (bf16 KV only)
  int fuse, L, T;
  const int32_t* slot_table;
  const __nv_bfloat16* q;
  const __nv_bfloat16* uk;
  const __nv_bfloat16* uv;
  __nv_bfloat16* out;
  // e4m3 KV: the unshared rows are read as fp8 by the fused epilogue (the
  // prompt KV reaches the tensor cores as bf16) and the output takes v_scale
  int kv8;
  const uint8_t* uk8;
  const uint8_t* uv8;
  const float* v_scale;
};

// Low word of a 128-byte-swizzle shared-memory descriptor (start address and
// leading byte offset, 16-byte units); the high word (stride byte offset,
// version 1, swizzle mode) is the same for every operand of this kernel.  The
// ring and Q lie below 256 KB, so a byte offset added to the address adds
// offset >> 4 to the low word without a carry out of its 14-bit field.
__device__ __forceinline__ uint32_t desc_lo(uint32_t addr, uint32_t lbo) {
  return ((addr & 0x3FFFFu) >> 4) | (((lbo & 0x3FFFFu) >> 4) << 16);
}
constexpr uint32_t desc_hi(uint32_t sbo) { return ((sbo & 0x3FFFFu) >> 4) | (1u << 14) | (2u << 29); }
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 da, db;\n setp.ne.b32 p, %5, 0;\n"
      " mov.b64 da, {%1, %3};\n mov.b64 db, {%2, %3};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, p;\n}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t hi,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 db;\n setp.ne.b32 p, %4, 0;\n"
      " mov.b64 db, {%2, %5};\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(hi));
}

struct Bars {
  uint64_t q;
  uint64_t kv_full[kSlots], kv_empty[kSlots];
  uint64_t s_full[2], p_full[2];
  uint64_t done;
  uint64_t probe;   // never completed: the timeout test hook waits on it
  uint64_t drain;   // an aborting MMA thread's last commit
};

// One lane polls (bounded), the warp agrees, then every lane observes the
// completed phase itself before touching the data it guards.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  bool ok = false;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok) ok = mbar_wait(bar, parity, 1u << 10);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool warp_flag(volatile int* f) {
  return __shfl_sync(0xffffffffu, *f, 0) != 0;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
      "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
      "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---- packed fp32 pairs: one f32x2 instruction does two lanes' worth --------
using f2 = unsigned long long;
__device__ __forceinline__ f2 f2_pack(float a, float b) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(f2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ f2 f2_fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// P = 2^(s * sc - m) for the 128 scores of one row as bf16 pairs into TMEM
// columns 0-63 of the row's S tile, and its sum (two f32x2 chains).  Every
// exponential is the MUFU ex2: moving some of them onto the FMA pipe (a
// range-reduced polynomial) measured slower here, because the softmax warps
// are short of issue slots as much as of MUFU throughput.
__device__ __forceinline__ void softmax_row(const float (&sv)[128], float sc, float m_used,
                                            uint32_t tS, f2& acc0, f2& acc1) {
  const f2 scv = f2_pack(sc, sc), nm = f2_pack(-m_used, -m_used);
#pragma unroll
  for (int q = 0; q < 4; ++q) {   // keys 32q .. 32q+31 -> columns 16q .. 16q+15
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int k2 = q * 32 + 2 * i;
      const f2 x = f2_fma(f2_pack(sv[k2], sv[k2 + 1]), scv, nm);
      const float2 xv = f2_unpack(x);
      const f2 pp = f2_pack(ex2(xv.x), ex2(xv.y));
      if (i & 1) acc1 = f2_add(acc1, pp);
      else acc0 = f2_add(acc0, pp);
      const float2 pv = f2_unpack(pp);
      const __nv_bfloat162 b = __floats2bfloat162_rn(pv.x, pv.y);
      pk[i] = *reinterpret_cast<const uint32_t*>(&b);
    }
    tmem_st16u(tS + 16 * q, pk);
  }
}

__device__ __forceinline__ void write_empty_partials(const TcParams& p, size_t base, int row0) {
  for (int i = threadIdx.x; i < 256; i += blockDim.x) {
    const int row = row0 + i;
    if (row >= p.rows) continue;
    p.pm[base + row] = -INFINITY;
    p.pl[base + row] = 0.f;
    float4* o = reinterpret_cast<float4*>(p.po + (base + row) * 128);
    for (int c = 0; c < 32; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t bf_pack(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Output row of query row `row` of (request r, kv head g): beam j = row / G,
// query head g * G + row % G.
__device__ __forceinline__ size_t out_row(const TcParams& p, int r, int g, int row) {
  const int j = row / p.G, h = row - j * p.G;
  return (((size_t)r * p.W + j) * p.Hq + (size_t)g * p.G + h) * 128;
}

// One unshared K row (128 elements, bf16 or e4m3 unscaled: the K scale is in
// the softmax scale) dotted with the query row, from the CTA's swizzled Q
// tile or from global memory when qtile is null.
__device__ __forceinline__ float unshared_dot(const TcParams& p, size_t e, const unsigned char* qtile, int rit,
                                              size_t qoff) {
  float d0 = 0.f, d1 = 0.f;
  auto qword = [&](int c) -> uint4 {   // bf16 query elements 8c .. 8c + 7
    return qtile ? *reinterpret_cast<const uint4*>(qtile + (c >> 3) * kHalfBytes + rit * 128 +
                                                   (((c & 7) ^ (rit & 7)) << 4))
                 : __ldg(reinterpret_cast<const uint4*>(p.q + qoff) + c);
  };
  if (p.kv8) {
    const uint4* kr = reinterpret_cast<const uint4*>(p.uk8 + e);
    uint4 kw[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) kw[c] = __ldg(kr + c);
#pragma unroll
    for (int c = 0; c < 8; ++c) {   // 16 key elements per 16-byte word
      const uint32_t w4[4] = {kw[c].x, kw[c].y, kw[c].z, kw[c].w};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 qw = qword(2 * c + h);
        const uint32_t qv[4] = {qw.x, qw.y, qw.z, qw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t kk = w4[2 * h + (i >> 1)] >> (16 * (i & 1));
          const float2 kf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(
              (__nv_fp8x2_storage_t)(kk & 0xffffu), __NV_E4M3)));
          d0 = fmaf(bf_lo(qv[i]), kf.x, d0);
          d1 = fmaf(bf_hi(qv[i]), kf.y, d1);
        }
      }
    }
  } else {
    const uint4* kr = reinterpret_cast<const uint4*>(p.uk + e);
    uint4 kw[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) kw[c] = __ldg(kr + c);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 qw = qword(c);
      d0 = fmaf(bf_lo(qw.x), bf_lo(kw[c].x), d0);
      d1 = fmaf(bf_hi(qw.x), bf_hi(kw[c].x), d1);
      d0 = fmaf(bf_lo(qw.y), bf_lo(kw[c].y), d0);
      d1 = fmaf(bf_hi(qw.y), bf_hi(kw[c].y), d1);
      d0 = fmaf(bf_lo(qw.z), bf_lo(kw[c].z), d0);
      d1 = fmaf(bf_hi(qw.z), bf_hi(kw[c].z), d1);
      d0 = fmaf(bf_lo(qw.w), bf_lo(kw[c].w), d0);
      d1 = fmaf(bf_hi(qw.w), bf_hi(kw[c].w), d1);
    }
  }
  return d0 + d1;
}

// o += w x (unshared V row e, columns q4*32 .. q4*32 + 31; e4m3 unscaled).
__device__ __forceinline__ void unshared_axpy(const TcParams& p, size_t e, int q4, float w, float (&o)[32]) {
  if (p.kv8) {
    const uint4* vr = reinterpret_cast<const uint4*>(p.uv8 + e + q4 * 32);
    const uint4 v0 = __ldg(vr), v1 = __ldg(vr + 1);
    const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(
          (__nv_fp8x2_storage_t)((wv[i >> 1] >> (16 * (i & 1))) & 0xffffu), __NV_E4M3)));
      o[2 * i] = fmaf(w, f.x, o[2 * i]);
      o[2 * i + 1] = fmaf(w, f.y, o[2 * i + 1]);
    }
  } else {
    const uint4* vr = reinterpret_cast<const uint4*>(p.uv + e + q4 * 32);
    uint4 vw[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) vw[c] = __ldg(vr + c);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      o[8 * c + 0] = fmaf(w, bf_lo(vw[c].x), o[8 * c + 0]);
      o[8 * c + 1] = fmaf(w, bf_hi(vw[c].x), o[8 * c + 1]);
      o[8 * c + 2] = fmaf(w, bf_lo(vw[c].y), o[8 * c + 2]);
      o[8 * c + 3] = fmaf(w, bf_hi(vw[c].y), o[8 * c + 3]);
      o[8 * c + 4] = fmaf(w, bf_lo(vw[c].z), o[8 * c + 4]);
      o[8 * c + 5] = fmaf(w, bf_hi(vw[c].z), o[8 * c + 5]);
      o[8 * c + 6] = fmaf(w, bf_lo(vw[c].w), o[8 * c + 6]);
      o[8 * c + 7] = fmaf(w, bf_hi(vw[c].w), o[8 * c + 7]);
    }
  }
}

// Fused epilogue, one query row per thread: the unshared stage over the
// beam's decode tokens (reached through its slot-table row; each K row is
// scored with the shared stage's log2-unit scale) and the online-softmax
// merge with the shared stage's (m, l, O):
//     M = max(m, s_u),  Lsum = l 2^(m - M) + sum_u 2^(s_u - M),
//     out = (O 2^(m - M) + sum_u 2^(s_u - M) v_u) / Lsum,
// written as bf16.  Dead beams' rows are written as zeros.  Every lane of a
// warp calls it (the TMEM loads of O are warp-wide).  have_o: O, m and l
// come from this CTA's shared stage; otherwise the prompt is empty.  The
// query row comes from the CTA's swizzled Q tile, or from global memory
// when qtile is null.  ps: scratch in shared memory, stride 128 words.
// The epilogue runs once per CTA, so its instructions are fetched cold: one
// token's loads at a time (a small body) measured faster than unrolled
// batches of tokens, and than half-warps sharing rows with shuffles.
__device__ __forceinline__ void fused_row(const TcParams& p, int r, int g, int row,
                                         const unsigned char* qtile, int rit, uint32_t tO,
                                         bool have_o, float m_used, float l, float sc, float* ps) {
  const int j = row / p.G;
  const bool in = row < p.rows;
  const bool live = in && j < p.n_live[r];
  const int L = p.L, TW = p.T * p.W;
  const bool shared_ok = have_o && l > 0.f;
  float M = shared_ok ? m_used : -INFINITY;
  const size_t qoff = in ? out_row(p, r, g, row) : 0;
  int* pslot = reinterpret_cast<int*>(ps + (size_t)L * 128);
  for (int u = 0; u < L; ++u) {
    int sl = live ? __ldg(p.slot_table + ((size_t)r * p.W + j) * p.T + u) : -1;
    if (live && (sl < 0 || sl >= TW)) {
      set_status(p.hdr, BEAMDEC_ERR_DEVICE_CHECK);
      sl = -1;
    }
    float s = -INFINITY;
    if (sl >= 0) s = unshared_dot(p, (((size_t)r * TW + sl) * p.Hkv + g) * 128, qtile, rit, qoff) * sc;
    ps[u * 128] = s;
    pslot[u * 128] = sl;
    M = fmaxf(M, s);
  }
  const float a = shared_ok ? ex2(m_used - M) : 0.f;
  float Ls = shared_ok ? l * a : 0.f;
  for (int u = 0; u < L; ++u) {
    const float w = pslot[u * 128] >= 0 ? ex2(ps[u * 128] - M) : 0.f;
    ps[u * 128] = w;
    Ls += w;
  }
  const float vs = (p.kv8 && p.v_scale) ? p.v_scale[g] : 1.f;   // e4m3 V is unscaled up to here
  const float inv = Ls > 0.f ? vs / Ls : 0.f;
#pragma unroll 1
  for (int q4 = 0; q4 < 4; ++q4) {
    float o[32];
    if (have_o) tmem_ld32(tO + q4 * 32, o);
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = shared_ok ? o[i] * a : 0.f;
    for (int u = 0; u < L; ++u) {
      const int sl = pslot[u * 128];
      if (sl < 0) continue;
      unshared_axpy(p, (((size_t)r * TW + sl) * p.Hkv + g) * 128, q4, ps[u * 128], o);
    }
    if (in) {
      uint4* dst = reinterpret_cast<uint4*>(p.out + qoff + q4 * 32);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        dst[c] = live ? make_uint4(bf_pack(o[8 * c] * inv, o[8 * c + 1] * inv),
                                   bf_pack(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                   bf_pack(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                   bf_pack(o[8 * c + 6] * inv, o[8 * c + 7] * inv))
                      : make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// Zero output rows [row0, row0 + 256) of (request r, kv head g): a CTA whose
// beams are all dead, when the merge is fused.
__device__ __forceinline__ void zero_rows(const TcParams& p, int r, int g, int row0) {
  for (int i = threadIdx.x; i < 256 * 16; i += blockDim.x) {
    const int row = row0 + (i >> 4);
    if (row < p.rows) reinterpret_cast<uint4*>(p.out + out_row(p, r, g, row))[i & 15] = make_uint4(0, 0, 0, 0);
  }
}

// Wait for the grid this one depends on (returns at once when there is none).
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// CTAs are dispatched in block-index order with blockIdx.z slowest, so the
// z-th plane of the grid takes the request with the z-th longest prompt
// (ties by index): the longest requests start first and the short ones fill
// the SMs behind them.  Up to 32 requests are ranked (one per lane, every
// warp the same); more keep the index order.
__device__ __forceinline__ int request_by_length(const int32_t* off, int R, int z) {
  if (R > 32) return z;
  const int lane = threadIdx.x & 31;
  const int len = lane < R ? off[lane + 1] - off[lane] : -1;
  int rank = 0;
  for (int j = 0; j < R; ++j) {
    const int lj = __shfl_sync(0xffffffffu, len, j);
    rank += (lj > len || (lj == len && j < lane)) ? 1 : 0;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, lane < R && rank == z);
  return hit ? __ffs(hit) - 1 : z;
}

// Eleven warps: the register file is handed out in groups of four warps, so a
// thread may hold at most 65536 / 384 -> 168 registers (a tenth or eleventh
// warp costs no registers).
__global__ void __launch_bounds__(kThreads, 1)
bd_attn_shared_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                         const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, TcParams p) {
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  // the timeout test hook (0 in normal use), loaded with the CTA's first
  // loads so that its latency hides behind theirs
  const uint32_t probe = *reinterpret_cast<volatile uint32_t*>(&p.hdr->probe_polls);
  const int mt = blockIdx.x;
  const int g = blockIdx.y % p.Hkv;
  const int sp = blockIdx.y / p.Hkv;
  const int r = request_by_length(p.prompt_offsets, p.R, blockIdx.z);
  const int row0 = mt * 256;
  const int G = p.G;
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) {
    if ((int64_t)p.prompt_offsets[p.R] != p.shared_rows)
      set_status(p.hdr, BEAMDEC_ERR_DEVICE_CHECK);   // the K/V maps end at shared_rows
    if (p.prep_k != nullptr &&
        (p.hdr->prep_k != reinterpret_cast<uintptr_t>(p.prep_k) ||
         p.hdr->prep_v != reinterpret_cast<uintptr_t>(p.prep_v) ||
         p.hdr->prep_rows != (unsigned long long)p.shared_rows ||
         p.hdr->prep_dst != reinterpret_cast<uintptr_t>(p.prep_dst)))
      set_status(p.hdr, BEAMDEC_ERR_DEVICE_CHECK);   // no copy of this prompt K/V at this place
  }
  if (!p.dep_wait_late) grid_dep_wait();
  if (!p.dep_wait_late && row0 >= p.n_live[r] * G) {   // every row of the CTA is a dead beam
    if (p.fuse) zero_rows(p, r, g, row0);
    return;
  }
  const int pbase = p.prompt_offsets[r];
  const int P = p.prompt_offsets[r + 1] - pbase;
  const int k0 = sp * p.split_len;
  const int k1 = min(P, k0 + p.split_len);
  const size_t prow_base = (((size_t)sp * p.R + r) * p.Hkv + g) * p.rows;
  if (k1 <= k0) {   // this split holds no key of the request
    if (!p.fuse) {
      write_empty_partials(p, prow_base, row0);
      if (threadIdx.x == 0) grid_dep_wait();   // this grid ends after the previous one
    } else if (threadIdx.x < 256) {   // empty prompt: the unshared tokens alone
      grid_dep_wait();
      const int t = threadIdx.x >> 7, rit = threadIdx.x & 127;
      float* ps = reinterpret_cast<float*>(sm + kOffKV + (uint32_t)t * (128u * 512u)) + rit;
      fused_row(p, r, g, row0 + threadIdx.x, nullptr, rit, 0u, false, -INFINITY, 0.f,
                p.scale_log2 * (p.k_scale ? p.k_scale[g] : 1.f), ps);
    }
    return;
  }
  const int nchunks = (k1 - k0 + 127) / 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&bars.q, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars.kv_full[s], 1);
      mbar_init(&bars.kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], 128);
    }
    mbar_init(&bars.done, 1);
    mbar_init(&bars.probe, 1);
    mbar_init(&bars.drain, 1);
    mbar_fence_init();
  }
  if (warp == 9) tmem_alloc(&tmem_base_sh, kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  if (probe != 0u) {   // test hook (block-uniform): a wait that runs out
    if (threadIdx.x == 0 && !mbar_wait(&bars.probe, 0, probe)) abort_sh = 1;
    __syncthreads();
  }

  if (abort_sh) {
    // nothing was issued: straight to the timeout exit
  } else if (warp == 8 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    const int j0 = row0 / G, jt = 128 / G;
    mbar_expect_tx(&bars.q, 2 * kTileBytes);
    tma_load_4d(sm + kOffQ, &qmap, &bars.q, 0, g * G, j0, r);
    tma_load_4d(sm + kOffQ + kHalfBytes, &qmap, &bars.q, 64, g * G, j0, r);
    tma_load_4d(sm + kOffQ + kTileBytes, &qmap, &bars.q, 0, g * G, j0 + jt, r);
    tma_load_4d(sm + kOffQ + kTileBytes + kHalfBytes, &qmap, &bars.q, 64, g * G, j0 + jt, r);
    int issued = 0;
    for (int i = 0; i < 2 * nchunks; ++i) {   // K0 V0 K1 V1 ...
      const int s = i % kSlots;
      const uint32_t u = (uint32_t)(i / kSlots);
      if (!mbar_wait(&bars.kv_empty[s], (u & 1) ^ 1)) { abort_sh = 1; break; }
      const int key = pbase + k0 + (i >> 1) * 128;
      const CUtensorMap* map = (i & 1) ? &vmap : &kmap;
      unsigned char* dst = sm + kOffKV + s * kTileBytes;
      mbar_expect_tx(&bars.kv_full[s], kTileBytes);
      tma_load_3d(dst, map, &bars.kv_full[s], 0, g, key);
      tma_load_3d(dst + kHalfBytes, map, &bars.kv_full[s], 64, g, key);
      issued = i + 1;
      if (abort_sh) break;
    }
    if (abort_sh) {   // let every copy this thread started land before exiting
      mbar_wait(&bars.q, 0);
      for (int i = (issued > kSlots ? issued - kSlots : 0); i < issued; ++i)
        mbar_wait(&bars.kv_full[i % kSlots], (uint32_t)(i / kSlots) & 1);
    }
  } else if (warp == 9 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    const uint32_t idO = idesc_bf16_f32(128, 128, false, true);
    const uint32_t qa = smem_u32(sm + kOffQ);
    const uint32_t kvb = smem_u32(sm + kOffKV);
    auto wait_kv = [&](int i) -> bool {
      return mbar_wait(&bars.kv_full[i % kSlots], (uint32_t)(i / kSlots) & 1);
    };
    const uint32_t hi = desc_hi(1024);   // Q, K and V: 8-row groups 1024 bytes apart
    const uint32_t q_lo = desc_lo(qa, 16), k_lo = desc_lo(kvb, 16), v_lo = desc_lo(kvb, kVLbo);
    auto issue_s = [&](int t, int c) {   // S_t = Q_t K(c)^T
      const uint32_t kb = k_lo + (uint32_t)((2 * c) % kSlots) * (kTileBytes >> 4);
      const uint32_t qt = q_lo + (uint32_t)t * (kTileBytes >> 4);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t off = ((k >> 2) * kHalfBytes + (k & 3) * 32) >> 4;
        mma_ss(tmem + t * 256, qt + off, kb + off, hi, idS, k > 0);
      }
      mma_commit(&bars.s_full[t]);
    };
    auto issue_pv = [&](int t, int c) {   // O_t += P_t V(c), P_t read from TMEM
      const uint32_t vb = v_lo + (uint32_t)((2 * c + 1) % kSlots) * (kTileBytes >> 4);
#pragma unroll
      for (int k = 0; k < 8; ++k)   // 16 keys = 8 columns of packed bf16 pairs per step
        mma_ts(tmem + t * 256 + 128, tmem + t * 256 + k * 8, vb + ((k * 16 * 128) >> 4), hi, idO,
               (c > 0 || k > 0) ? 1u : 0u);
    };
    bool ok = mbar_wait(&bars.q, 0) && wait_kv(0);
    if (ok) {
      fence_after_sync();
      issue_s(0, 0);
      issue_s(1, 0);
      mma_commit(&bars.kv_empty[0]);
    }
    for (int c = 0; ok && c < nchunks; ++c) {
      const bool more = c + 1 < nchunks;
      if (!wait_kv(2 * c + 1)) { ok = false; break; }                 // V(c)
      if (!mbar_wait(&bars.p_full[0], c & 1)) { ok = false; break; }
      fence_after_sync();
      issue_pv(0, c);
      if (more) {   // p_full also says S_0(c) has been read
        if (!wait_kv(2 * c + 2)) { ok = false; break; }               // K(c+1)
        issue_s(0, c + 1);
      }
      if (!mbar_wait(&bars.p_full[1], c & 1)) { ok = false; break; }
      fence_after_sync();
      issue_pv(1, c);
      mma_commit(&bars.kv_empty[(2 * c + 1) % kSlots]);               // V(c) consumed
      if (more) {
        issue_s(1, c + 1);
        mma_commit(&bars.kv_empty[(2 * c + 2) % kSlots]);             // K(c+1) consumed
      }
      if (abort_sh) { ok = false; break; }
    }
    if (ok) {
      mma_commit(&bars.done);
    } else {
      abort_sh = 1;
      // the MMAs already issued complete before the CTA frees TMEM and exits
      mma_commit(&bars.drain);
      mbar_wait(&bars.drain, 0);
    }
  } else if (warp == 10 && p.fuse) {
    // ------------------------------------------------------------ L2 prefetch
    // pulls this CTA's unshared K/V rows into L2 while the shared stage runs,
    // so the fused epilogue reads them from L2
    grid_dep_wait();
    const int TW = p.T * p.W, nb = 256 / G, j0 = row0 / G, nl = p.n_live[r];
    for (int i = lane; i < nb * p.L; i += 32) {
      const int jj = i / p.L, u = i - jj * p.L;
      const int j = j0 + jj;
      if (j >= nl) continue;
      const int sl = __ldg(p.slot_table + ((size_t)r * p.W + j) * p.T + u);
      if (sl < 0 || sl >= TW) continue;
      const size_t e = (((size_t)r * TW + sl) * p.Hkv + g) * 128;
      if (p.kv8) {
        bulk_prefetch_l2(p.uk8 + e, 128);
        bulk_prefetch_l2(p.uv8 + e, 128);
      } else {
        bulk_prefetch_l2(p.uk + e, 256);
        bulk_prefetch_l2(p.uv + e, 256);
      }
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax rows
    const int t = warp >> 2;                       // tile
    const int row_in_tile = threadIdx.x - t * 128;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + t * 256 + lane_off;
    const uint32_t tO = tS + 128;
    const float sc = p.scale_log2 * (p.k_scale ? p.k_scale[g] : 1.f);
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      if (!warp_wait(&bars.s_full[t], c & 1)) { ok = false; break; }
      fence_after_sync();
      // pass 1: the chunk's row max (one 128-column TMEM load); only the last
      // chunk of a split can hold fewer than 128 keys, so the full case runs
      // without per-element masks
      const int nvalid = min(128, k1 - (k0 + c * 128));
      const bool full = nvalid == 128;
      float mx = -INFINITY;
      {
        float sv[128];
        tmem_ld128(tS, sv);
        if (full) {   // tree of three-input maxima: 128 -> 43 -> 15 -> 5 -> 1
#pragma unroll
          for (int i = 0; i < 42; ++i) sv[i] = max3f(sv[3 * i], sv[3 * i + 1], sv[3 * i + 2]);
          sv[42] = fmaxf(sv[126], sv[127]);
#pragma unroll
          for (int i = 0; i < 14; ++i) sv[i] = max3f(sv[3 * i], sv[3 * i + 1], sv[3 * i + 2]);
          sv[14] = sv[42];
#pragma unroll
          for (int i = 0; i < 5; ++i) sv[i] = max3f(sv[3 * i], sv[3 * i + 1], sv[3 * i + 2]);
          mx = max3f(sv[0], sv[1], max3f(sv[2], sv[3], sv[4]));
        } else {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i < nvalid) mx = fmaxf(mx, sv[i]);
        }
      }
      mx *= sc;
      const bool need = mx > m_used + kRescale;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_used;
        const float factor = ex2(m_used - m_new);   // 0 on the first chunk, 1 for rows that keep m
        l *= factor;
        if (c > 0) {   // O_t holds chunks < c (their PV completed before S_t(c) was signalled)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float v[32];
            tmem_ld32(tO + q * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= factor;
            tmem_st32(tO + q * 32, v);
          }
          tmem_wait_st();
        }
        m_used = m_new;
      }
      // pass 2: P = 2^(s - m) as bf16 pairs into TMEM columns 0-63 of S_t
      // (the last, partial chunk masks its missing keys: ex2 gives exact zeros)
      f2 acc0 = f2_pack(0.f, 0.f), acc1 = f2_pack(0.f, 0.f);
      {
        float sv[128];
        tmem_ld128(tS, sv);
        if (!full) {
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= nvalid) sv[i] = -INFINITY;
        }
        softmax_row(sv, sc, m_used, tS, acc0, acc1);
      }
      {
        const float2 a0 = f2_unpack(acc0), a1 = f2_unpack(acc1);
        l += (a0.x + a0.y) + (a1.x + a1.y);
      }
      tmem_wait_st();
      fence_before_sync();
      mbar_arrive(&bars.p_full[t]);
      if (warp_flag(&abort_sh)) { ok = false; break; }
    }
    if (ok && !warp_wait(&bars.done, 0)) ok = false;
    if (!ok) abort_sh = 1;
    const int row = row0 + t * 128 + row_in_tile;
    if (p.fuse) {   // unshared stage + merge here; the K/V ring is idle now
      grid_dep_wait();
      if (ok) {
        fence_after_sync();
        float* ps = reinterpret_cast<float*>(sm + kOffKV + (uint32_t)t * (128u * 512u)) + row_in_tile;
        fused_row(p, r, g, row, sm + kOffQ + t * kTileBytes, row_in_tile, tO, true, m_used, l, sc, ps);
      }
    } else {
      // O_t leaves through shared memory (the K/V ring is idle once every MMA
      // is done): each thread puts its row there, 16-byte chunks swizzled by
      // the row, then each warp stores whole 512-byte rows, coalesced
      unsigned char* stage = sm + kOffKV + (uint32_t)t * (128u * 512u);
      if (ok) {
        fence_after_sync();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[32];
          tmem_ld32(tO + q * 32, v);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int chunk = q * 8 + i;
            *reinterpret_cast<float4*>(stage + row_in_tile * 512 + ((chunk ^ (row_in_tile & 7)) << 4)) =
                make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          }
        }
      }
      named_bar(1 + t, 128);   // the tile's four warps; every one of them arrives, ok or not
      if (ok) {
        for (int rr = warp & 3; rr < 128; rr += 4) {
          const int grow = row0 + t * 128 + rr;
          if (grow < p.rows) {
            const float4 v = *reinterpret_cast<const float4*>(stage + rr * 512 + ((lane ^ (rr & 7)) << 4));
            reinterpret_cast<float4*>(p.po + (prow_base + grow) * 128)[lane] = v;
          }
        }
        if (row < p.rows) {
          p.pm[prow_base + row] = m_used;
          p.pl[prow_base + row] = l;
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (abort_sh && threadIdx.x == 0) set_status(p.hdr, BEAMDEC_ERR_TIMEOUT);
  // Whatever the path, one thread of every CTA waits for the previous grid
  // before exiting, so this grid completes only after that one: the kernels
  // after it in the stream (the merge kernel reads the slot table) keep the
  // ordinary stream order.
  if (threadIdx.x == 0) grid_dep_wait();
  if (warp == 9) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// fp8 e4m3 K/V of the prompt -> bf16 (exact: every e4m3 value is a bf16
// value), rows [0, prompt_offsets[R]), for the tensor-core shared stage.  The
// per-head scales are not applied here: K's scale multiplies the softmax
// scale and V's scale the merged output.
// It reads nothing the selection writes, so it is launched as a programmatic
// dependent of the previous kernel; inside a decode call it lets the shared
// stage launch the same way (that stage waits for this grid before its main
// loop), while beam_attn_prepare_prompt's copy does not (a prepared call
// reads the copy without waiting).  Each thread waits for the previous grid
// before it exits, so that this grid's completion implies that one's.
__global__ void __launch_bounds__(256)
bd_kv_e4m3_to_bf16_kernel(const uint8_t* __restrict__ k8, const uint8_t* __restrict__ v8,
                          __nv_bfloat16* __restrict__ k16, __nv_bfloat16* __restrict__ v16,
                          const int32_t* prompt_offsets, int R, int64_t row_elems, WsHeader* hdr,
                          int64_t shared_rows, int early) {
  if (early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0 && threadIdx.x == 0) {   // what the copy holds, for prepared calls
    hdr->prep_k = reinterpret_cast<uintptr_t>(k8);
    hdr->prep_v = reinterpret_cast<uintptr_t>(v8);
    hdr->prep_rows = (unsigned long long)shared_rows;
    hdr->prep_dst = reinterpret_cast<uintptr_t>(k16);
  }
  const int64_t n16 = (int64_t)prompt_offsets[R] * row_elems / 16;   // 16-element groups
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < 2 * n16;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool isv = i >= n16;
    const int64_t e = (isv ? i - n16 : i) * 16;
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>((isv ? v8 : k8) + e));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[q] >> (16 * h)) & 0xffffu);
        const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
        const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
        o[2 * q + h] = *reinterpret_cast<const uint32_t*>(&b);
      }
    }
    uint4* dst = reinterpret_cast<uint4*>((isv ? v16 : k16) + e);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
  grid_dep_wait();
}

// ---- host side ------------------------------------------------------------------

// Launch with programmatic stream serialization (the kernel may begin before
// the previous kernel in the stream completes, when that kernel allows it).
template <class... P, class... A>
cudaError_t launch_dependent(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}
}  // namespace

bool attn_tc_supported(int q_dtype, int kv_dtype, int d, int G) {
  return q_dtype == BEAMDEC_BF16 && (kv_dtype == BEAMDEC_BF16 || kv_dtype == BEAMDEC_E4M3) &&
         d == 128 && G >= 1 && G <= 16 && (128 % G) == 0;
}

// The merge runs in the shared stage's epilogue when the whole prompt is one
// split (every query row's shared partial stays in its CTA), the KV is bf16
// or e4m3 (the epilogue reads e4m3 unshared rows as fp8 and scales the output
// by v_scale), the unshared tokens fit the epilogue's scratch and the rows
// are 16-byte aligned for vector loads and stores.
bool attn_tc_fused(const AttnArgs& a, const AttnPlan& pl) {
  const auto al16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  return pl.tensor_core && pl.n_split == 1 && (a.kv_dtype == BEAMDEC_BF16 || a.kv_dtype == BEAMDEC_E4M3) &&
         a.out_dtype == BEAMDEC_BF16 &&
         a.d == 128 && a.step + 1 <= kFusedMaxL && al16(a.q) && al16(a.unshared_k) && al16(a.unshared_v) &&
         al16(a.out);
}

int launch_kv_copy(const AttnArgs& a, const AttnPlan& pl, cudaStream_t stream, bool early) {
  __nv_bfloat16* k16 = attn_kv16(a.ws, a.R, a.W, a.Hq, a.Hkv, a.d, pl.n_split);
  __nv_bfloat16* v16 = k16 + (size_t)a.R * a.max_prompt_len * a.Hkv * a.d;
  const int64_t groups = a.shared_rows * a.Hkv * a.d / 16 * 2;
  int blocks = (int)((groups + 255) / 256);
  if (blocks > 8 * sm_count()) blocks = 8 * sm_count();
  if (blocks < 1) blocks = 1;
  prof_begin(kKKvConvert, stream);
  const cudaError_t ce = launch_dependent(bd_kv_e4m3_to_bf16_kernel, dim3(blocks), dim3(256), 0, stream,
                                          static_cast<const uint8_t*>(a.shared_k),
                                          static_cast<const uint8_t*>(a.shared_v), k16, v16, a.prompt_offsets,
                                          a.R, (int64_t)a.Hkv * a.d, reinterpret_cast<WsHeader*>(a.ws),
                                          a.shared_rows, early ? 1 : 0);
  prof_end(kKKvConvert, stream);
  return (ce == cudaSuccess && cudaGetLastError() == cudaSuccess) ? BEAMDEC_OK : BEAMDEC_ERR_CUDA;
}

int launch_attn_shared_tc(const AttnArgs& a, const AttnPlan& pl, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  if (!attn_tc_supported(a.q_dtype, a.kv_dtype, a.d, G)) return BEAMDEC_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(a.q) & 15) || (reinterpret_cast<uintptr_t>(a.shared_k) & 15) ||
      (reinterpret_cast<uintptr_t>(a.shared_v) & 15))
    return BEAMDEC_ERR_INVALID_ARG;
  static PerDeviceOnce attr_once;
  const int arc = once_per_device(attr_once, [](int) {
    return cudaFuncSetAttribute(bd_attn_shared_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemBytes) == cudaSuccess ? BEAMDEC_OK : BEAMDEC_ERR_CUDA;
  });
  if (arc != BEAMDEC_OK) return arc;
  // with no prompt key at all (shared_rows = 0, K/V may be NULL) the K/V
  // maps are never loaded from; they are encoded over the queries' memory,
  // which holds at least one [Hkv][d] row, so that the encode sees a valid
  // address
  const void* kbase = a.shared_rows > 0 ? a.shared_k : a.q;
  const void* vbase = a.shared_rows > 0 ? a.shared_v : a.q;
  if (a.kv_dtype == BEAMDEC_E4M3 && a.shared_rows > 0) {
    // the prompt KV as bf16 in the workspace: made here, or earlier by
    // beam_attn_prepare_prompt
    if (!a.kv_prepared) {
      const int rc = launch_kv_copy(a, pl, stream, true);
      if (rc != BEAMDEC_OK) return rc;
    }
    __nv_bfloat16* k16 = attn_kv16(a.ws, a.R, a.W, a.Hq, a.Hkv, a.d, pl.n_split);
    kbase = k16;
    vbase = k16 + (size_t)a.R * a.max_prompt_len * a.Hkv * a.d;
  }
  CUtensorMap qm, km, vm;
  {
    const cuuint64_t dims[4] = {(cuuint64_t)a.d, (cuuint64_t)a.Hq, (cuuint64_t)a.W, (cuuint64_t)a.R};
    const cuuint64_t st[3] = {(cuuint64_t)a.d * 2, (cuuint64_t)a.Hq * a.d * 2,
                              (cuuint64_t)a.W * a.Hq * a.d * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G), 1};
    if (!make_map(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.q, dims, st, box)) return BEAMDEC_ERR_CUDA;
  }
  {
    const cuuint64_t total = (cuuint64_t)a.shared_rows;   // rows allocated in shared_k / shared_v
    const cuuint64_t dims[3] = {(cuuint64_t)a.d, (cuuint64_t)a.Hkv, total > 0 ? total : 1};
    const cuuint64_t st[2] = {(cuuint64_t)a.d * 2, (cuuint64_t)a.Hkv * a.d * 2};
    const cuuint32_t box[3] = {64, 1, 128};
    if (!make_map(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kbase, dims, st, box) ||
        !make_map(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, vbase, dims, st, box))
      return BEAMDEC_ERR_CUDA;
  }
  TcParams p;
  p.R = a.R; p.W = a.W; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.rows = a.W * G;
  p.split_len = pl.split_len;
  p.scale_log2 = a.sm_scale * kLog2e;
  p.k_scale = a.kv_dtype == BEAMDEC_E4M3 ? a.k_scale : nullptr;
  p.shared_rows = a.shared_rows;
  p.prompt_offsets = a.prompt_offsets;
  p.n_live = a.n_live;
  AttnPartials part = attn_partials(a.ws, a.R, a.W, a.Hq, a.Hkv, a.d, pl.n_split);
  p.pm = part.m; p.pl = part.l; p.po = part.o;
  p.hdr = reinterpret_cast<WsHeader*>(a.ws);
  p.fuse = attn_tc_fused(a, pl) ? 1 : 0;
  p.L = a.step + 1;
  p.T = a.T;
  p.slot_table = a.slot_table;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.uk = static_cast<const __nv_bfloat16*>(a.unshared_k);
  p.uv = static_cast<const __nv_bfloat16*>(a.unshared_v);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.kv8 = a.kv_dtype == BEAMDEC_E4M3 ? 1 : 0;
  p.uk8 = static_cast<const uint8_t*>(a.unshared_k);
  p.uv8 = static_cast<const uint8_t*>(a.unshared_v);
  p.v_scale = a.kv_dtype == BEAMDEC_E4M3 ? a.v_scale : nullptr;
  dim3 grid((p.rows + 255) / 256, a.Hkv * pl.n_split, a.R);
  prof_begin(kKAttnTc, stream);
  // A programmatic dependent of the previous kernel in the stream: its CTAs
  // may start while that kernel drains, if it allows it (the selection's
  // kernels do).  The main loop reads only Q and the prompt K/V; the slot
  // table and the live counts are read after the previous grid completes.
  // At step 0 (one live beam per request) the CTAs wait first, so that
  // dead tiles skip the main loop; the bf16 copy of e4m3 K/V is waited for
  // before the main loop too.
  p.dep_wait_late = (a.step > 0 && !(a.kv_dtype == BEAMDEC_E4M3 && a.shared_rows > 0 && !a.kv_prepared)) ? 1 : 0;
  p.prep_k = (a.kv_prepared && a.shared_rows > 0) ? a.shared_k : nullptr;
  p.prep_v = a.shared_v;
  p.prep_dst = kbase;
  const cudaError_t le = launch_dependent(bd_attn_shared_tc_kernel, grid, dim3(kThreads), kSmemBytes, stream,
                                          qm, km, vm, p);
  prof_end(kKAttnTc, stream);
  return le == cudaSuccess && cudaGetLastError() == cudaSuccess ? BEAMDEC_OK : BEAMDEC_ERR_CUDA;
}

}  // namespace bd
