// LM-head GEMM with the log-sum-exp fused into its epilogue.
//
// The step before the selection: logits = hidden x W^T over the whole
// vocabulary.  "Generative recommendation design" (xLLM) §4.3 filters invalid
// item paths before they become candidates; here the full-vocabulary logits
// are reduced to each row's log-sum-exp inside the GEMM, and only a window of
// token columns (the current SID level's code range) is written out, so the
// [rows, V] logits never reach HBM.  The selection then runs on that window
// with the row normalisers passed in (beam_select with lse_in).
//
// A persistent grid (one CTA per SM) walks the 128-row x 256-column output
// tiles, row tiles fastest so that the CTAs running together share one slab
// of W in L2:
//   warp 0       TMA producer: 64-wide K slabs of hidden (128 x 64) and W
//                (256 x 64), SWIZZLE_128B, through a 4-stage ring that runs
//                on across tiles;
//   warp 1       allocates 512 TMEM columns (two 256-column accumulators)
//                and issues the kind::f16 MMAs (M 128, N 256, K 16; bf16 in,
//                fp32 accumulate) of tile i into accumulator i % 2;
//   warps 2-5    epilogue, one row per thread (TMEM lane), on the other
//                accumulator meanwhile: the tile's (max, sum of exp) in log2
//                units per row, and the window columns stored through a
//                shared-memory staging chunk in coalesced row segments.
// A second kernel folds each row's per-tile partials into its log-sum-exp.
// Every mbarrier wait is bounded; a timeout records BEAMDEC_ERR_TIMEOUT, the
// other roles stop at their next wait, the copies in flight land and TMEM
// is still freed.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace bd {
namespace {

using namespace tc;

constexpr int kLmThreads = 192;
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;              // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;              // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kOutChunkBytes = kBM * 64 * 4;        // 32 KB: 64 fp32 columns of 128 rows
constexpr uint32_t kLmSmem = kStages * kStageBytes + kOutChunkBytes + 1024;

struct LmParams {
  int rows, hidden, V, n_tiles, m_tiles, win0, win1;
  int64_t out_stride;
  float* out;        // window logits (may be null when the window is empty)
  float2* part;      // [rows][n_tiles] (max, sum of 2^(x - max)), log2 units
  WsHeader* hdr;
};

struct LmBars {
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t probe;   // never completed: the timeout test hook waits on it
  uint64_t drain;   // an aborting MMA thread's last commit
};

__device__ __forceinline__ bool warp_flag(volatile int* f) {
  return __shfl_sync(0xffffffffu, *f, 0) != 0;
}

__device__ __forceinline__ bool warp_wait_lm(uint64_t* bar, uint32_t parity) {
  bool ok = false;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok) ok = mbar_wait(bar, parity, 1u << 10);
  return __all_sync(0xffffffffu, ok);
}

__global__ void __launch_bounds__(kLmThreads, 1)
bd_lmhead_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                 LmParams p) {
  extern __shared__ __align__(1024) unsigned char dsm_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
  __shared__ LmBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the timeout test hook (0 in normal use), loaded first so that its
  // latency hides behind the set-up below
  const uint32_t probe = *reinterpret_cast<volatile uint32_t*>(&p.hdr->probe_polls);
  const int nk = p.hidden / kBK;
  const int total = p.m_tiles * p.n_tiles;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars.full[s], 1);
      mbar_init(&bars.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&bars.acc_full[a], 1);
      mbar_init(&bars.acc_empty[a], 128);
    }
    mbar_init(&bars.probe, 1);
    mbar_init(&bars.drain, 1);
    mbar_fence_init();
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, 2 * kBN);
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
  } else if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    prefetch_tmap(&amap);
    prefetch_tmap(&bmap);
    uint32_t g = 0, issued = 0;
    for (int t = blockIdx.x; t < total && !abort_sh; t += gridDim.x) {
      const int row0 = (t % p.m_tiles) * kBM, col0 = (t / p.m_tiles) * kBN;
      for (int k = 0; k < nk; ++k, ++g) {
        const int s = (int)(g % kStages);
        if (!mbar_wait(&bars.empty[s], ((g / kStages) & 1u) ^ 1u)) { abort_sh = 1; break; }
        unsigned char* dst = sm + s * kStageBytes;
        mbar_expect_tx(&bars.full[s], kStageBytes);
        tma_load_2d(dst, &amap, &bars.full[s], k * kBK, row0);
        tma_load_2d(dst + kABytes, &bmap, &bars.full[s], k * kBK, col0);
        issued = g + 1;
      }
    }
    if (abort_sh) {   // let every copy this thread started land before exiting
      for (uint32_t i = (issued > (uint32_t)kStages ? issued - kStages : 0); i < issued; ++i)
        mbar_wait(&bars.full[i % kStages], (i / kStages) & 1u);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(kBM, kBN, false, false);
    const uint32_t base = smem_u32(sm);
    uint32_t g = 0;
    int i = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++i) {
      const int acc = i & 1;
      if (!mbar_wait(&bars.acc_empty[acc], ((uint32_t)(i >> 1) & 1u) ^ 1u)) { ok = false; break; }
      fence_after_sync();
      const uint32_t d = tmem + acc * kBN;
      for (int k = 0; k < nk; ++k, ++g) {
        const int s = (int)(g % kStages);
        if (!mbar_wait(&bars.full[s], (g / kStages) & 1u)) { ok = false; break; }
        fence_after_sync();
        const uint32_t a0 = base + s * kStageBytes, b0 = a0 + kABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk)
          mma_bf16(d, sdesc_sw128(a0 + kk * 32, 16, 1024), sdesc_sw128(b0 + kk * 32, 16, 1024), idesc,
                   (k > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars.empty[s]);   // the slot is free once these MMAs have read it
      }
      if (!ok) break;
      mma_commit(&bars.acc_full[acc]);
      if (abort_sh) ok = false;
    }
    if (!ok) {
      abort_sh = 1;
      // the MMAs already issued complete before the CTA frees TMEM and exits
      mma_commit(&bars.drain);
      mbar_wait(&bars.drain, 0);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane group of this warp
    const int srow = q * 32 + lane;               // row inside the tile
    float* stage = reinterpret_cast<float*>(sm + kStages * kStageBytes);   // [128][64]
    int i = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
      const int acc = i & 1;
      const int row0 = (t % p.m_tiles) * kBM, col0 = (t / p.m_tiles) * kBN;
      const int row = row0 + srow;
      // every epilogue warp runs the same barrier sequence; a timeout only
      // skips the work
      bool ok = !warp_flag(&abort_sh) && warp_wait_lm(&bars.acc_full[acc], (uint32_t)(i >> 1) & 1u);
      if (!ok) abort_sh = 1;
      if (ok) fence_after_sync();
      const uint32_t taddr = tmem + acc * kBN + ((uint32_t)(q * 32) << 16);
      const bool win_tile = p.out != nullptr && col0 < p.win1 && col0 + kBN > p.win0;
      float m = -INFINITY, l = 0.f;
#pragma unroll 1
      for (int c = 0; c < kBN / 64; ++c) {
        const int cb = col0 + c * 64;
        float v[64];
        if (ok) {
          tmem_ld64(taddr + c * 64, v);
          float mc = -INFINITY;
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (cb + j < p.V) mc = fmaxf(mc, v[j]);
          mc *= kLog2e;
          const float mn = fmaxf(m, mc);
          float sum = 0.f;
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (cb + j < p.V) sum += ex2(fmaf(v[j], kLog2e, -mn));
          l = (l > 0.f ? l * ex2(m - mn) : 0.f) + sum;
          m = mn;
        }
        if (win_tile && cb < p.win1 && cb + 64 > p.win0) {   // uniform over the epilogue warps
          if (ok) {
#pragma unroll
            for (int j4 = 0; j4 < 16; ++j4)
              reinterpret_cast<float4*>(stage + srow * 64)[j4 ^ (srow & 15)] =
                  make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
          }
          named_bar(1, 128);
          if (ok) {
            const int c_lo = max(p.win0, cb), c_hi = min(min(p.win1, p.V), cb + 64);
            for (int rr = q * 32; rr < q * 32 + 32; ++rr) {
              const int grow = row0 + rr;
              if (grow >= p.rows) break;
              const int cc = c_lo + lane;   // 64 columns: two per lane
              float* orow = p.out + (int64_t)grow * p.out_stride;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int col = cc + 32 * h;
                if (col < c_hi) {
                  const int j = col - cb;
                  orow[col] = stage[rr * 64 + (((j >> 2) ^ (rr & 15)) << 2) + (j & 3)];
                }
              }
            }
          }
          named_bar(1, 128);   // the chunk buffer is free again
        }
      }
      // this accumulator's TMEM reads are complete (tcgen05.wait::ld): hand it back
      fence_before_sync();
      mbar_arrive(&bars.acc_empty[acc]);
      if (ok && row < p.rows) p.part[(int64_t)row * p.n_tiles + (t / p.m_tiles)] = make_float2(m, l);
    }
  }
  fence_before_sync();
  __syncthreads();
  if (abort_sh && threadIdx.x == 0) set_status(p.hdr, BEAMDEC_ERR_TIMEOUT);
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, 2 * kBN);
  }
}

// One warp per row: fold the row's per-tile (max, sum) into its log-sum-exp.
__global__ void __launch_bounds__(256)
bd_lmhead_lse_kernel(const float2* __restrict__ part, int rows, int n_tiles, float* __restrict__ lse) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= rows) return;
  float m = -INFINITY, l = 0.f;
  for (int i = lane; i < n_tiles; i += 32) {
    const float2 t = part[(int64_t)row * n_tiles + i];
    if (!(t.y > 0.f)) continue;
    const float mn = fmaxf(m, t.x);
    l = (l > 0.f ? l * ex2(m - mn) : 0.f) + t.y * ex2(t.x - mn);
    m = mn;
  }
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), l2 = __shfl_xor_sync(0xffffffffu, l, o);
    const float mn = fmaxf(m, m2);
    const float a = l > 0.f ? l * ex2(m - mn) : 0.f, b = l2 > 0.f ? l2 * ex2(m2 - mn) : 0.f;
    m = mn;
    l = a + b;
  }
  if (lane == 0) lse[row] = (m + log2f(l)) * 0.69314718055994531f;
}

}  // namespace

size_t lmhead_workspace_bytes(int rows, int V) {
  const int n_tiles = (V + kBN - 1) / kBN;
  return kWsHeaderBytes + (size_t)rows * n_tiles * sizeof(float2);
}

int launch_lmhead(const void* hidden, const void* weight, int rows, int hidden_dim, int V,
                  int win0, int win1, float* lse_out, float* logits_out, int64_t out_stride,
                  void* ws, cudaStream_t stream) {
  static PerDeviceOnce attr_once;
  const int arc = once_per_device(attr_once, [](int) {
    return cudaFuncSetAttribute(bd_lmhead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kLmSmem) == cudaSuccess ? BEAMDEC_OK : BEAMDEC_ERR_CUDA;
  });
  if (arc != BEAMDEC_OK) return arc;
  CUtensorMap am, bm;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)hidden_dim, (cuuint64_t)rows};
    const cuuint64_t st[1] = {(cuuint64_t)hidden_dim * 2};
    const cuuint32_t box[2] = {kBK, kBM};
    if (!make_map(&am, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, hidden, dims, st, box)) return BEAMDEC_ERR_CUDA;
  }
  {
    const cuuint64_t dims[2] = {(cuuint64_t)hidden_dim, (cuuint64_t)V};
    const cuuint64_t st[1] = {(cuuint64_t)hidden_dim * 2};
    const cuuint32_t box[2] = {kBK, kBN};
    if (!make_map(&bm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, weight, dims, st, box)) return BEAMDEC_ERR_CUDA;
  }
  LmParams p;
  p.rows = rows; p.hidden = hidden_dim; p.V = V;
  p.n_tiles = (V + kBN - 1) / kBN;
  p.m_tiles = (rows + kBM - 1) / kBM;
  p.win0 = win0; p.win1 = win1;
  p.out = logits_out; p.out_stride = out_stride;
  p.hdr = reinterpret_cast<WsHeader*>(ws);
  p.part = reinterpret_cast<float2*>(static_cast<char*>(ws) + kWsHeaderBytes);
  const int tiles = p.m_tiles * p.n_tiles;
  dim3 grid(tiles < sm_count() ? tiles : sm_count());
  prof_begin(kKLmhead, stream);
  bd_lmhead_kernel<<<grid, kLmThreads, kLmSmem, stream>>>(am, bm, p);
  prof_end(kKLmhead, stream);
  if (cudaGetLastError() != cudaSuccess) return BEAMDEC_ERR_CUDA;
  prof_begin(kKLmheadLse, stream);
  bd_lmhead_lse_kernel<<<(rows + 7) / 8, 256, 0, stream>>>(p.part, rows, p.n_tiles, lse_out);
  prof_end(kKLmheadLse, stream);
  return cudaGetLastError() == cudaSuccess ? BEAMDEC_OK : BEAMDEC_ERR_CUDA;
}

}  // namespace bd
