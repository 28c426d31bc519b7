// Shared stage of the beam attention on the tcgen05 tensor cores.
//
// "Generative recommendation design" (xLLM) §4.2.1-§4.2.2: the prompt KV of a
// request is stored once and all of its beams attend to it, so for one
// (request, kv head g) the queries of every beam and every query head of the
// group form one dense matrix Q [W*G x d] against the prompt's K and V: the
// shared stage is a flash-attention contraction with M = W*G rows.  Its
// output is the partial (max, sum, unnormalised output) of every query row,
// merged later with the unshared stage.
//
// One CTA owns 128 query rows of one (request, kv head, prompt split):
//   warp 0      TMA producer: Q once, then K and V tiles of 128 keys
//               (two 64-column SWIZZLE_128B boxes each) into a 2-stage ring;
//   warp 1      allocates TMEM and issues the MMAs from one thread:
//               S = Q K^T (M 128, N 128, K 128) into a double-buffered TMEM
//               score tile, and O_c = P V (M 128, N 128, K 128; V read
//               d-major) into a double-buffered TMEM output tile;
//   warps 4-7   softmax: thread t owns query row t (TMEM lane t); reads its
//               scores from TMEM, keeps the running max / sum in log2 units,
//               writes P as bf16 into shared memory in the 128B-swizzled
//               K-major layout the MMA reads, and folds each chunk's output
//               O_c into a register accumulator one chunk behind the MMAs.
// Every wait on an mbarrier is bounded; a timeout records
// BEAMDEC_ERR_TIMEOUT, stops the loops and still frees TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace bd {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr uint32_t kHalfBytes = 16384;          // 128 rows x 128 B
constexpr uint32_t kTileBytes = 2 * kHalfBytes; // 128 x 128 bf16
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kTileBytes;                 // 2 stages
constexpr uint32_t kOffV = kOffK + 2 * kTileBytes;     // 2 stages
constexpr uint32_t kOffP = kOffV + 2 * kTileBytes;
constexpr uint32_t kSmemBytes = kOffP + kTileBytes + 1024;  // + alignment slack
constexpr uint32_t kTmemCols = 512;  // S0 S1 O0 O1, 128 columns each

// MN-major B operand (V, d contiguous): the leading byte offset is the stride
// between 64-column swizzle atoms along d (the two 16 KB halves), the stride
// byte offset the stride between groups of 8 keys (8 x 128 B).
constexpr uint32_t kVLbo = kHalfBytes;
constexpr uint32_t kVSbo = 1024;

struct TcParams {
  int R, W, Hq, Hkv, G, rows, split_len;
  float scale_log2;   // sm_scale * log2(e)
  const int32_t* prompt_offsets;
  const int32_t* n_live;
  const float* k_scale;   // fp8 only (nullptr otherwise)
  float* pm;
  float* pl;
  float* po;
  WsHeader* hdr;
};

struct Bars {
  uint64_t q;
  uint64_t full_k[2], empty_k[2], full_v[2], empty_v[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, pv_done;
};

// One lane polls (bounded), the warp agrees on the outcome, then every lane
// observes the completed phase itself (acquire) before touching the data.
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

__device__ __forceinline__ void write_empty_partials(const TcParams& p, size_t base, int row0, int nrows) {
  for (int i = threadIdx.x; i < 128; i += blockDim.x) {
    const int row = row0 + i;
    if (row >= nrows) continue;
    p.pm[base + row] = -INFINITY;
    p.pl[base + row] = 0.f;
    float4* o = reinterpret_cast<float4*>(p.po + (base + row) * 128);
    for (int c = 0; c < 32; ++c) o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
bd_attn_shared_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                         const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, TcParams p) {
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* sm =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;

  const int mt = blockIdx.x;
  const int g = blockIdx.y % p.Hkv;
  const int sp = blockIdx.y / p.Hkv;
  const int r = blockIdx.z;
  const int row0 = mt * 128;
  const int G = p.G;
  if (row0 >= p.n_live[r] * G) return;   // every row of the tile is a dead beam
  const int pbase = p.prompt_offsets[r];
  const int P = p.prompt_offsets[r + 1] - pbase;
  const int k0 = sp * p.split_len;
  const int k1 = min(P, k0 + p.split_len);
  const size_t pbase_rows = ((size_t)sp * p.R + r) * p.Hkv + g;
  const size_t prow_base = pbase_rows * p.rows;
  if (k1 <= k0) {   // this split holds no key of the request
    write_empty_partials(p, prow_base, row0, p.rows);
    return;
  }
  const int nchunks = (k1 - k0 + 127) / 128;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    mbar_init(&bars.q, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars.full_k[s], 1);
      mbar_init(&bars.empty_k[s], 1);
      mbar_init(&bars.full_v[s], 1);
      mbar_init(&bars.empty_v[s], 1);
      mbar_init(&bars.s_full[s], 1);
      mbar_init(&bars.s_free[s], 128);
    }
    mbar_init(&bars.p_full, 128);
    mbar_init(&bars.pv_done, 1);
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    prefetch_tmap(&qmap);
    prefetch_tmap(&kmap);
    prefetch_tmap(&vmap);
    const int j0 = row0 / G;
    mbar_expect_tx(&bars.q, kTileBytes);
    tma_load_4d(sm + kOffQ, &qmap, &bars.q, 0, g * G, j0, r);
    tma_load_4d(sm + kOffQ + kHalfBytes, &qmap, &bars.q, 64, g * G, j0, r);
    int issued = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      const uint32_t ph = (c >> 1) & 1;
      const int key = pbase + k0 + c * 128;
      if (!mbar_wait(&bars.empty_k[s], ph ^ 1)) { abort_sh = 1; break; }
      mbar_expect_tx(&bars.full_k[s], kTileBytes);
      tma_load_3d(sm + kOffK + s * kTileBytes, &kmap, &bars.full_k[s], 0, g, key);
      tma_load_3d(sm + kOffK + s * kTileBytes + kHalfBytes, &kmap, &bars.full_k[s], 64, g, key);
      if (!mbar_wait(&bars.empty_v[s], ph ^ 1)) { abort_sh = 1; issued = c * 2 + 1; break; }
      mbar_expect_tx(&bars.full_v[s], kTileBytes);
      tma_load_3d(sm + kOffV + s * kTileBytes, &vmap, &bars.full_v[s], 0, g, key);
      tma_load_3d(sm + kOffV + s * kTileBytes + kHalfBytes, &vmap, &bars.full_v[s], 64, g, key);
      issued = c * 2 + 2;
      if (abort_sh) break;
    }
    if (abort_sh) {
      // let every copy this thread started land before the CTA exits
      mbar_wait(&bars.q, 0);
      for (int u = 0; u < issued; ++u) {
        const int c = u >> 1, s = c & 1;
        mbar_wait((u & 1) ? &bars.full_v[s] : &bars.full_k[s], (c >> 1) & 1);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idS = idesc_bf16_f32(128, 128, false, false);
    const uint32_t idO = idesc_bf16_f32(128, 128, false, true);
    const uint32_t qa = smem_u32(sm + kOffQ);
    bool ok = mbar_wait(&bars.q, 0);
    auto issue_s = [&](int c) -> bool {
      const int s = c & 1;
      if (!mbar_wait(&bars.full_k[s], (c >> 1) & 1)) return false;
      if (!mbar_wait(&bars.s_free[s], ((c >> 1) & 1) ^ 1)) return false;
      fence_after_sync();
      const uint32_t kb = smem_u32(sm + kOffK + s * kTileBytes);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t off = (k >> 2) * kHalfBytes + (k & 3) * 32;
        mma_bf16(tmem + s * 128, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024), idS,
                 k > 0);
      }
      mma_commit(&bars.empty_k[s]);
      mma_commit(&bars.s_full[s]);
      return true;
    };
    if (ok) ok = issue_s(0);
    for (int c = 0; ok && c < nchunks; ++c) {
      if (c + 1 < nchunks && !issue_s(c + 1)) { ok = false; break; }
      const int s = c & 1;
      if (!mbar_wait(&bars.p_full, c & 1)) { ok = false; break; }
      if (!mbar_wait(&bars.full_v[s], (c >> 1) & 1)) { ok = false; break; }
      fence_after_sync();
      const uint32_t pa = smem_u32(sm + kOffP);
      const uint32_t vb = smem_u32(sm + kOffV + s * kTileBytes);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint64_t a = sdesc_sw128(pa + (k >> 2) * kHalfBytes + (k & 3) * 32, 16, 1024);
        const uint32_t vk = vb + k * 16 * 128;   // 16 keys per step
        mma_bf16(tmem + 256 + s * 128, a, sdesc_sw128(vk, kVLbo, kVSbo), idO, k > 0);
      }
      mma_commit(&bars.empty_v[s]);
      mma_commit(&bars.pv_done);
      if (abort_sh) { ok = false; break; }
    }
    if (!ok) abort_sh = 1;
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax rows
    const int t = threadIdx.x - 128;           // query row within the tile = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp - 4) * 32) << 16;
    const float ks = p.k_scale ? p.k_scale[g] : 1.f;
    const float sc = p.scale_log2 * ks;
    float m = -INFINITY, l = 0.f, alpha_prev = 1.f;
    float O[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) O[i] = 0.f;
    unsigned char* Ps = sm + kOffP;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      if (!warp_wait(&bars.s_full[s], (c >> 1) & 1)) { ok = false; break; }
      fence_after_sync();
      const int nvalid = min(128, k1 - (k0 + c * 128));
      float mx = -INFINITY;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[32];
        tmem_ld32(tmem + s * 128 + lane_off + q * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (q * 32 + i < nvalid) mx = fmaxf(mx, v[i]);
      }
      const float m_new = fmaxf(m, mx * sc);
      const float alpha = ex2(m - m_new);
      if (c > 0) {
        if (!warp_wait(&bars.pv_done, (c - 1) & 1)) { ok = false; break; }
        fence_after_sync();
      }
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float v[32];
        tmem_ld32(tmem + s * 128 + lane_off + q * 32, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int k2 = q * 32 + 2 * i;
          const float p0 = (k2 < nvalid) ? ex2(fmaf(v[2 * i], sc, -m_new)) : 0.f;
          const float p1 = (k2 + 1 < nvalid) ? ex2(fmaf(v[2 * i + 1], sc, -m_new)) : 0.f;
          const __nv_bfloat162 b = __floats2bfloat162_rn(p0, p1);
          const float2 bf = __bfloat1622float2(b);
          sum += bf.x + bf.y;
          pk[i] = *reinterpret_cast<const uint32_t*>(&b);
        }
        const int half = q >> 1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int chunk = (q & 1) * 4 + k;
          uint4* dst = reinterpret_cast<uint4*>(Ps + half * kHalfBytes + t * 128 +
                                                ((chunk ^ (t & 7)) << 4));
          *dst = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        }
      }
      fence_before_sync();
      mbar_arrive(&bars.s_free[s]);
      fence_proxy_async_smem();
      mbar_arrive(&bars.p_full);
      l = l * alpha + sum;
      if (c > 0) {   // fold O of the previous chunk (its PV is complete)
        const int so = (c - 1) & 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[32];
          tmem_ld32(tmem + 256 + so * 128 + lane_off + q * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) O[q * 32 + i] = fmaf(O[q * 32 + i], alpha_prev, v[i]);
        }
      }
      alpha_prev = alpha;
      m = m_new;
      if (warp_flag(&abort_sh)) { ok = false; break; }
    }
    if (ok) {
      if (warp_wait(&bars.pv_done, (nchunks - 1) & 1)) {
        fence_after_sync();
        const int so = (nchunks - 1) & 1;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[32];
          tmem_ld32(tmem + 256 + so * 128 + lane_off + q * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) O[q * 32 + i] = fmaf(O[q * 32 + i], alpha_prev, v[i]);
        }
      } else {
        ok = false;
      }
    }
    if (!ok) abort_sh = 1;
    const int row = row0 + t;
    if (ok && row < p.rows) {
      const size_t pi = prow_base + row;
      p.pm[pi] = m;
      p.pl[pi] = l;
      float4* o = reinterpret_cast<float4*>(p.po + pi * 128);
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = make_float4(O[4 * i], O[4 * i + 1], O[4 * i + 2], O[4 * i + 3]);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (abort_sh && threadIdx.x == 0) set_status(p.hdr, BEAMDEC_ERR_TIMEOUT);
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- host side ------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base,
              const cuuint64_t* dims, const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides_bytes, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool attn_tc_supported(int q_dtype, int kv_dtype, int d, int G) {
  return q_dtype == BEAMDEC_BF16 && kv_dtype == BEAMDEC_BF16 && d == 128 && G >= 1 && G <= 16 &&
         (128 % G) == 0;
}

int launch_attn_shared_tc(const AttnArgs& a, const AttnPlan& pl, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  if (!attn_tc_supported(a.q_dtype, a.kv_dtype, a.d, G)) return BEAMDEC_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(a.q) & 15) || (reinterpret_cast<uintptr_t>(a.shared_k) & 15) ||
      (reinterpret_cast<uintptr_t>(a.shared_v) & 15))
    return BEAMDEC_ERR_INVALID_ARG;
  static bool attr_set[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BEAMDEC_ERR_CUDA;
  if (!attr_set[dev]) {
    if (cudaFuncSetAttribute(bd_attn_shared_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
      return BEAMDEC_ERR_CUDA;
    attr_set[dev] = true;
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
    if (!make_map(&km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.shared_k, dims, st, box) ||
        !make_map(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.shared_v, dims, st, box))
      return BEAMDEC_ERR_CUDA;
  }
  TcParams p;
  p.R = a.R; p.W = a.W; p.Hq = a.Hq; p.Hkv = a.Hkv; p.G = G; p.rows = a.W * G;
  p.split_len = pl.split_len;
  p.scale_log2 = a.sm_scale * kLog2e;
  p.prompt_offsets = a.prompt_offsets;
  p.n_live = a.n_live;
  p.k_scale = nullptr;
  AttnPartials part = attn_partials(a.ws, a.R, a.W, a.Hq, a.Hkv, a.d, pl.n_split);
  p.pm = part.m; p.pl = part.l; p.po = part.o;
  p.hdr = reinterpret_cast<WsHeader*>(a.ws);
  dim3 grid((p.rows + 127) / 128, a.Hkv * pl.n_split, a.R);
  prof_begin(kKAttnTc, stream);
  bd_attn_shared_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(qm, km, vm, p);
  prof_end(kKAttnTc, stream);
  return cudaGetLastError() == cudaSuccess ? BEAMDEC_OK : BEAMDEC_ERR_CUDA;
}

}  // namespace bd
