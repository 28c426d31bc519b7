// Unshared stage and online-softmax merge of the beam attention.
//
// "Generative recommendation design" (xLLM) §4.2.1: the decode tokens of each
// beam live in the unshared KV, one entry per token, addressed here through
// the parent-pointer slot table (beam reorder copies slot indices, never KV);
// §4.2.2: the unshared stage computes its own partial (max, sum, output) and
// the merge combines it with the shared stage's partials:
//     M = max_i m_i,  L = sum_i l_i 2^(m_i - M),  O = sum_i o_i 2^(m_i - M),
//     out = v_scale * O / L
// (scores are kept in log2 units: the softmax scale is pre-multiplied by
// log2 e, so 2^x replaces e^x exactly in value).
//
// One warp per (request, beam, query head).  Lane l owns dims
// [l*D/32, (l+1)*D/32).  The beam's slot row (<= 32 entries read per step) is
// loaded once, one slot per lane, and broadcast with shuffles.  Loads that do
// not depend on each other (query, the first splits' partials, a few tokens'
// K and V) are issued together so a warp waits on few memory round trips.
#include <cuda_runtime.h>
#include <math.h>

#include "attn_common.cuh"
#include "common.cuh"
#include "internal.h"

namespace bd {
namespace {

template <int DT, int PL>
__device__ __forceinline__ void load_lane(const void* base, size_t e, float (&x)[PL]) {
  if constexpr (PL == 4) {
    const float4 v = load4<DT>(base, e);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  } else {
    // PL == 2: two elements; read the enclosing 4-aligned group and pick a half
    const size_t e4 = e & ~(size_t)3;
    const float4 v = load4<DT>(base, e4);
    if (e == e4) { x[0] = v.x; x[1] = v.y; } else { x[0] = v.z; x[1] = v.w; }
  }
}

template <int DQ, int DKV, int D>
__global__ void __launch_bounds__(512, 2)
bd_attn_merge_kernel(AttnArgs a, int n_split, AttnPartials part) {
  constexpr int PL = D / 32;
  constexpr int kPre = 2;          // prompt splits whose partials are prefetched
  constexpr int kTok = PL == 4 ? 2 : 4;   // unshared tokens whose K/V loads are in flight together
  const int j = blockIdx.x, r = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int G = a.Hq / a.Hkv;
  const int rows = a.W * G;
  const bool live = j < a.n_live[r];
  WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
  const int L = a.step + 1;
  const int TW = a.T * a.W;
  int my_slot = -1;
  if (live && lane < L) {
    my_slot = a.slot_table[((size_t)r * a.W + j) * a.T + lane];
    if (my_slot < 0 || my_slot >= TW) {
      set_status(hdr, BEAMDEC_ERR_DEVICE_CHECK);
      my_slot = -1;
    }
  }
  for (int h = threadIdx.x >> 5; h < a.Hq; h += nwarps) {
    const size_t out_e = (((size_t)r * a.W + j) * a.Hq + h) * D + lane * PL;
    if (!live) {
      if constexpr (PL == 4) {
        store_out4(a.out, out_e, make_float4(0.f, 0.f, 0.f, 0.f), a.out_dtype);
      } else {
        if (a.out_dtype == 0) {
          static_cast<float*>(a.out)[out_e] = 0.f;
          static_cast<float*>(a.out)[out_e + 1] = 0.f;
        } else {
          static_cast<__nv_bfloat16*>(a.out)[out_e] = __float2bfloat16(0.f);
          static_cast<__nv_bfloat16*>(a.out)[out_e + 1] = __float2bfloat16(0.f);
        }
      }
      continue;
    }
    const int g = h / G, gi = h - g * G;
    const int row = j * G + gi;
    // independent loads first: query, and the first splits' partial triples
    float q[PL];
    load_lane<DQ, PL>(a.q, out_e, q);
    float pm_l = -INFINITY, pl_l = 0.f;   // lane c holds split c's (m, l)
    if (lane < n_split) {
      const size_t pi = (((size_t)lane * a.R + r) * a.Hkv + g) * rows + row;
      pm_l = part.m[pi];
      pl_l = part.l[pi];
    }
    float oc[kPre][PL];
#pragma unroll
    for (int c = 0; c < kPre; ++c) {
      if (c < n_split) {
        const size_t pi = (((size_t)c * a.R + r) * a.Hkv + g) * rows + row;
        const float* src = part.o + pi * D + lane * PL;
        if constexpr (PL == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          oc[c][0] = v.x; oc[c][1] = v.y; oc[c][2] = v.z; oc[c][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          oc[c][0] = v.x; oc[c][1] = v.y;
        }
      } else {
#pragma unroll
        for (int i = 0; i < PL; ++i) oc[c][i] = 0.f;
      }
    }
    const float ks = (DKV == 2 && a.k_scale) ? a.k_scale[g] : 1.f;
    const float vs = (DKV == 2 && a.v_scale) ? a.v_scale[g] : 1.f;
    const float scale2 = a.sm_scale * kLog2e * ks;
#pragma unroll
    for (int i = 0; i < PL; ++i) q[i] *= scale2;
    // unshared stage over the beam's L decode tokens, kTok tokens per round
    float m = -INFINITY, l = 0.f, o[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) o[i] = 0.f;
    for (int t0 = 0; t0 < L; t0 += kTok) {
      int slot[kTok];
      float k[kTok][PL], v[kTok][PL];
#pragma unroll
      for (int u = 0; u < kTok; ++u) {
        const int t = t0 + u;
        int sl = __shfl_sync(0xffffffffu, my_slot, t & 31);
        if (t >= L) sl = -1;
        else if (t >= 32) {   // rows longer than a warp: read the entry directly
          sl = a.slot_table[((size_t)r * a.W + j) * a.T + t];
          if (sl < 0 || sl >= TW) {
            if (lane == 0) set_status(hdr, BEAMDEC_ERR_DEVICE_CHECK);
            sl = -1;
          }
        }
        slot[u] = sl;
        if (sl >= 0) {
          const size_t e = (((size_t)r * TW + sl) * a.Hkv + g) * D + lane * PL;
          load_lane<DKV, PL>(a.unshared_k, e, k[u]);
          load_lane<DKV, PL>(a.unshared_v, e, v[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < kTok; ++u) {
        if (slot[u] < 0) continue;
        float sdot = 0.f;
#pragma unroll
        for (int i = 0; i < PL; ++i) sdot = fmaf(q[i], k[u][i], sdot);
        sdot = warp_sum(sdot);
        const float mn = fmaxf(m, sdot);
        const float alpha = ex2(m - mn), pt = ex2(sdot - mn);
        l = l * alpha + pt;
#pragma unroll
        for (int i = 0; i < PL; ++i) o[i] = fmaf(pt, v[u][i], o[i] * alpha);
        m = mn;
      }
    }
    // merge with the shared-stage partials of every prompt split
    float M = m;
    for (int c = 0; c < n_split; ++c) {
      const float mc = c < 32 ? __shfl_sync(0xffffffffu, pm_l, c)
                              : part.m[(((size_t)c * a.R + r) * a.Hkv + g) * rows + row];
      M = fmaxf(M, mc);
    }
    const float wu = (l == 0.f) ? 0.f : ex2(m - M);
    float Lsum = l * wu;
    float O[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) O[i] = o[i] * wu;
    for (int c = 0; c < n_split; ++c) {
      const size_t pi = (((size_t)c * a.R + r) * a.Hkv + g) * rows + row;
      const float mc = c < 32 ? __shfl_sync(0xffffffffu, pm_l, c) : part.m[pi];
      const float lc = c < 32 ? __shfl_sync(0xffffffffu, pl_l, c) : part.l[pi];
      if (lc == 0.f) continue;
      const float w = ex2(mc - M);
      Lsum = fmaf(lc, w, Lsum);
      if (c < kPre) {
#pragma unroll
        for (int cc = 0; cc < kPre; ++cc)
          if (cc == c) {
#pragma unroll
            for (int i = 0; i < PL; ++i) O[i] = fmaf(oc[cc][i], w, O[i]);
          }
      } else {
        const float* src = part.o + pi * D + lane * PL;
#pragma unroll
        for (int i = 0; i < PL; ++i) O[i] = fmaf(src[i], w, O[i]);
      }
    }
    const float inv = vs / Lsum;
    if constexpr (PL == 4) {
      store_out4(a.out, out_e, make_float4(O[0] * inv, O[1] * inv, O[2] * inv, O[3] * inv),
                 a.out_dtype);
    } else {
      if (a.out_dtype == 0) {
        static_cast<float*>(a.out)[out_e] = O[0] * inv;
        static_cast<float*>(a.out)[out_e + 1] = O[1] * inv;
      } else {
        static_cast<__nv_bfloat16*>(a.out)[out_e] = __float2bfloat16_rn(O[0] * inv);
        static_cast<__nv_bfloat16*>(a.out)[out_e + 1] = __float2bfloat16_rn(O[1] * inv);
      }
    }
  }
}

template <int DQ, int DKV, int D>
int launch_t(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream) {
  int threads = 32 * (a.Hq < 16 ? a.Hq : 16);
  dim3 grid(a.W, a.R);
  AttnPartials part = attn_partials(a.ws, a.R, a.W, a.Hq, a.Hkv, a.d, p.n_split);
  prof_begin(kKAttnMerge, stream);
  bd_attn_merge_kernel<DQ, DKV, D><<<grid, threads, 0, stream>>>(a, p.n_split, part);
  prof_end(kKAttnMerge, stream);
  return cudaGetLastError() == cudaSuccess ? BEAMDEC_OK : BEAMDEC_ERR_CUDA;
}

}  // namespace

int launch_attn_merge(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream) {
  if (a.d == 128) {
    if (a.q_dtype == 0 && a.kv_dtype == 0) return launch_t<0, 0, 128>(a, p, stream);
    if (a.q_dtype == 1 && a.kv_dtype == 1) return launch_t<1, 1, 128>(a, p, stream);
    if (a.q_dtype == 1 && a.kv_dtype == 2) return launch_t<1, 2, 128>(a, p, stream);
  } else if (a.d == 64) {
    if (a.q_dtype == 0 && a.kv_dtype == 0) return launch_t<0, 0, 64>(a, p, stream);
    if (a.q_dtype == 1 && a.kv_dtype == 1) return launch_t<1, 1, 64>(a, p, stream);
    if (a.q_dtype == 1 && a.kv_dtype == 2) return launch_t<1, 2, 64>(a, p, stream);
  }
  return BEAMDEC_ERR_UNSUPPORTED;
}

}  // namespace bd
