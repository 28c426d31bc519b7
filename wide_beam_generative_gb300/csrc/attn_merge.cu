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
// One warp per (request, beam, kv head).  Lane l owns dims
// [l*D/32, (l+1)*D/32).  The beam's slot row (<= 32 entries read per step) is
// loaded once, one slot per lane, and broadcast with shuffles; each unshared
// K/V row is loaded once for all query heads of its group.  Loads that do
// not depend on each other (queries, partial (m, l), a few tokens' K and V)
// are issued together so a warp waits on few memory round trips.  Beams with
// 8 or more unshared tokens run the unshared stage in four groups of eight
// lanes (one token per group at a time, D/8 dims per lane), which cuts the
// shuffle steps of the per-token dot products; measured on 2 x 5000 beams
// with 32 tokens: decode step 2579 -> 2420 us.
#include <cuda_runtime.h>
#include <math.h>

#include <cuda_fp16.h>
#include <cuda_fp8.h>

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


// Raw storage of PL consecutive K/V elements of one lane, kept packed in
// 32-bit words until use (bf16: 2 per word, e4m3: 4 per word, fp32: 1).
template <int DT, int PL>
struct KvRaw {
  static constexpr int kWords = DT == 0 ? PL : (DT == 1 ? (PL + 1) / 2 : 1);
  uint32_t w[kWords];
  __device__ __forceinline__ void load(const void* base, size_t e) {
    if constexpr (DT == 0) {
      if constexpr (PL == 4) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + e));
        w[0] = __float_as_uint(v.x); w[1] = __float_as_uint(v.y);
        w[2] = __float_as_uint(v.z); w[3] = __float_as_uint(v.w);
      } else {
        const float2 v = __ldg(reinterpret_cast<const float2*>(static_cast<const float*>(base) + e));
        w[0] = __float_as_uint(v.x); w[1] = __float_as_uint(v.y);
      }
    } else if constexpr (DT == 1) {
      if constexpr (PL == 4) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + e));
        w[0] = v.x; w[1] = v.y;
      } else {
        w[0] = __ldg(reinterpret_cast<const unsigned int*>(static_cast<const __nv_bfloat16*>(base) + e));
      }
    } else {
      if constexpr (PL == 4) {
        w[0] = __ldg(reinterpret_cast<const unsigned int*>(static_cast<const uint8_t*>(base) + e));
      } else {
        w[0] = __ldg(reinterpret_cast<const unsigned short*>(static_cast<const uint8_t*>(base) + e));
      }
    }
  }
  __device__ __forceinline__ void to_float(float (&x)[PL]) const {
    if constexpr (DT == 0) {
#pragma unroll
      for (int i = 0; i < PL; ++i) x[i] = __uint_as_float(w[i]);
    } else if constexpr (DT == 1) {
#pragma unroll
      for (int i = 0; i < PL / 2; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < PL / 2; ++i) {
        const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[0] >> (16 * i)) & 0xffffu);
        const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
    }
  }
};

// N consecutive elements of one K/V row for a lane of an eight-lane group
// (N = D / 8), kept packed until use; 16-byte (e4m3 with N = 8: 8-byte)
// vector loads, so the tensor's base must be 16-byte aligned.
template <int DT, int N>
struct KvSlice {
  static constexpr int kWords = DT == 0 ? N : (DT == 1 ? N / 2 : N / 4);
  uint32_t w[kWords];
  __device__ __forceinline__ void load(const void* base, size_t e) {
    constexpr int es = DT == 0 ? 4 : (DT == 1 ? 2 : 1);
    const char* p = static_cast<const char*>(base) + e * es;
    if constexpr (kWords % 4 == 0) {
#pragma unroll
      for (int c = 0; c < kWords / 4; ++c) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p) + c);
        w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
      }
    } else {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
      w[0] = v.x; w[1] = v.y;
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = 0u;
  }
  __device__ __forceinline__ void to_float(float (&x)[N]) const {
    if constexpr (DT == 0) {
#pragma unroll
      for (int i = 0; i < N; ++i) x[i] = __uint_as_float(w[i]);
    } else if constexpr (DT == 1) {
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)((w[i >> 1] >> (16 * (i & 1))) & 0xffffu);
        const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3)));
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
    }
  }
};

// N consecutive query elements (fp32 or bf16) with 16-byte loads.
template <int DQ, int N>
__device__ __forceinline__ void load_q_slice(const void* base, size_t e, float (&x)[N]) {
  if constexpr (DQ == 0) {
#pragma unroll
    for (int c = 0; c < N / 4; ++c) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + e) + c);
      x[4 * c] = v.x; x[4 * c + 1] = v.y; x[4 * c + 2] = v.z; x[4 * c + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int c = 0; c < N / 8; ++c) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + e) + c);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
        x[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
      }
    }
  }
}

template <int DQ, int DKV, int D>
__device__ __forceinline__ void store_lane(void* out, size_t e, const float (&v)[D / 32], int out_dtype) {
  if constexpr (D / 32 == 4) {
    store_out4(out, e, make_float4(v[0], v[1], v[2], v[3]), out_dtype);
  } else {
    if (out_dtype == 0) {
      static_cast<float*>(out)[e] = v[0];
      static_cast<float*>(out)[e + 1] = v[1];
    } else {
      static_cast<__nv_bfloat16*>(out)[e] = __float2bfloat16_rn(v[0]);
      static_cast<__nv_bfloat16*>(out)[e + 1] = __float2bfloat16_rn(v[1]);
    }
  }
}

// One warp per (request, beam, kv head g), looping over the G query heads of
// the group in groups of kGq so each unshared K/V row is loaded once.
// kGrp (beams with 8 or more unshared tokens, 16-byte aligned tensors): the
// unshared stage runs in four groups of eight lanes, each group scoring one
// token at a time with D / 8 dims per lane, so a token's dot product needs
// three shuffle steps, shared by the group's token, instead of five for
// every token; the groups' partials are combined once at the end.
// Two 256-thread blocks per SM (up to 128 registers): at three (80
// registers) the whole-warp stage spilled about 280 bytes per thread and a
// 1 x 50 beam step took 46.0 us against 43.8 us.
template <int DQ, int DKV, int D, bool kGrp>
__global__ void __launch_bounds__(256, 2)
bd_attn_merge_kernel(AttnArgs a, int n_split, AttnPartials part) {
  constexpr int PL = D / 32;
  constexpr int kGq = 2;           // query heads per pass
  constexpr int kTok = 4;          // unshared tokens whose K/V loads are in flight together
  const int lane = threadIdx.x & 31;
  const int G = a.Hq / a.Hkv;
  const int rows = a.W * G;
  const int TW = a.T * a.W;
  const int L = a.step + 1;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
  const long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= (long long)a.R * a.W * a.Hkv) return;
  const int g = (int)(wid % a.Hkv);
  const int j = (int)((wid / a.Hkv) % a.W);
  const int r = (int)(wid / ((long long)a.Hkv * a.W));
  const size_t head0 = ((size_t)r * a.W + j) * a.Hq + (size_t)g * G;
  // first round of independent loads: live count, slot row, and below the
  // queries and partials of the first head group
  const int nl = a.n_live[r];
  int my_slot = lane < L ? a.slot_table[((size_t)r * a.W + j) * a.T + lane] : -1;
  const bool live = j < nl;
  if (!live) {
    float z[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) z[i] = 0.f;
    for (int gi = 0; gi < G; ++gi) store_lane<DQ, DKV, D>(a.out, (head0 + gi) * D + lane * PL, z, a.out_dtype);
    return;
  }
  if (lane < L && (my_slot < 0 || my_slot >= TW)) {
    set_status(hdr, BEAMDEC_ERR_DEVICE_CHECK);
    my_slot = -1;
  }
  const float ks = (DKV == 2 && a.k_scale) ? a.k_scale[g] : 1.f;
  const float vs = (DKV == 2 && a.v_scale) ? a.v_scale[g] : 1.f;
  const float scale2 = a.sm_scale * kLog2e * ks;
  for (int g0 = 0; g0 < G; g0 += kGq) {
    const int ng = G - g0 < kGq ? G - g0 : kGq;
    // independent loads: queries and the shared-stage partials of these heads
    float q[kGq][PL], o[kGq][PL], m[kGq], l[kGq], o0[kGq][PL];
    float pm[kGq], pl[kGq];   // lane c < n_split holds split c
#pragma unroll
    for (int u = 0; u < kGq; ++u) {
      m[u] = -INFINITY;
      l[u] = 0.f;
      pm[u] = -INFINITY;
      pl[u] = 0.f;
#pragma unroll
      for (int i = 0; i < PL; ++i) { q[u][i] = 0.f; o[u][i] = 0.f; o0[u][i] = 0.f; }
      if (u < ng) {
        load_lane<DQ, PL>(a.q, (head0 + g0 + u) * D + lane * PL, q[u]);
        if (n_split > 0) {   // split 0's partial output, prefetched
          const size_t p0 = (((size_t)r) * a.Hkv + g) * rows + (size_t)j * G + g0 + u;
          const float* src = part.o + p0 * D + lane * PL;
          if constexpr (PL == 4) {
            const float4 x = *reinterpret_cast<const float4*>(src);
            o0[u][0] = x.x; o0[u][1] = x.y; o0[u][2] = x.z; o0[u][3] = x.w;
          } else {
            const float2 x = *reinterpret_cast<const float2*>(src);
            o0[u][0] = x.x; o0[u][1] = x.y;
          }
        }
#pragma unroll
        for (int i = 0; i < PL; ++i) q[u][i] *= scale2;
        if (lane < n_split) {
          const size_t pi = (((size_t)lane * a.R + r) * a.Hkv + g) * rows + (size_t)j * G + g0 + u;
          pm[u] = part.m[pi];
          pl[u] = part.l[pi];
        }
      }
    }
    if constexpr (kGrp) {
      constexpr int N = D / 8;
      constexpr int kR = 1;   // tokens per group in flight
      const int grp = lane >> 3, gl = lane & 7;
      float qg[kGq][N], gm[kGq], gs[kGq], go[kGq][N];
#pragma unroll
      for (int u = 0; u < kGq; ++u) {
        gm[u] = -INFINITY;
        gs[u] = 0.f;
#pragma unroll
        for (int i = 0; i < N; ++i) { qg[u][i] = 0.f; go[u][i] = 0.f; }
        if (u < ng) load_q_slice<DQ, N>(a.q, (head0 + g0 + u) * D + gl * N, qg[u]);
#pragma unroll
        for (int i = 0; i < N; ++i) qg[u][i] *= scale2;
      }
      for (int t0 = 0; t0 < L; t0 += 4 * kR) {
        int sl[kR];
        KvSlice<DKV, N> kr[kR], vr[kR];
#pragma unroll
        for (int w = 0; w < kR; ++w) {
          const int t = t0 + 4 * w + grp;
          int s = __shfl_sync(0xffffffffu, my_slot, t & 31);
          if (t >= L) s = -1;
          else if (t >= 32) {   // rows longer than a warp: read the entry directly
            s = a.slot_table[((size_t)r * a.W + j) * a.T + t];
            if (s < 0 || s >= TW) {
              if (gl == 0) set_status(hdr, BEAMDEC_ERR_DEVICE_CHECK);
              s = -1;
            }
          }
          sl[w] = s;
          if (s >= 0) {
            const size_t e = (((size_t)r * TW + s) * a.Hkv + g) * D + gl * N;
            kr[w].load(a.unshared_k, e);
            vr[w].load(a.unshared_v, e);
          } else {
            kr[w].zero();
            vr[w].zero();
          }
        }
#pragma unroll
        for (int w = 0; w < kR; ++w) {
          float k[N];
          kr[w].to_float(k);
          float d[kGq];
#pragma unroll
          for (int u = 0; u < kGq; ++u) {
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int i = 0; i < N; i += 2) {
              d0 = fmaf(qg[u][i], k[i], d0);
              d1 = fmaf(qg[u][i + 1], k[i + 1], d1);
            }
            d[u] = d0 + d1;
          }
#pragma unroll
          for (int u = 0; u < kGq; ++u) {   // the group's eight lanes hold the token's partial sums
            d[u] += __shfl_xor_sync(0xffffffffu, d[u], 4);
            d[u] += __shfl_xor_sync(0xffffffffu, d[u], 2);
            d[u] += __shfl_xor_sync(0xffffffffu, d[u], 1);
          }
          if (sl[w] >= 0) {   // uniform in the group
            float v[N];
            vr[w].to_float(v);
#pragma unroll
            for (int u = 0; u < kGq; ++u) {
              if (u >= ng) continue;
              const float mn = fmaxf(gm[u], d[u]);
              const float alpha = ex2(gm[u] - mn), pt = ex2(d[u] - mn);
              gs[u] = gs[u] * alpha + pt;
#pragma unroll
              for (int i = 0; i < N; ++i) go[u][i] = fmaf(pt, v[i], go[u][i] * alpha);
              gm[u] = mn;
            }
          }
        }
      }
      // the four groups' (max, sum, output) -> one per head, laid out as the
      // whole-warp stage leaves it: lane l holds dims [PL l, PL l + PL)
#pragma unroll
      for (int u = 0; u < kGq; ++u) {
        float M = gm[u];
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 8));
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
        const float wg = gs[u] > 0.f ? ex2(gm[u] - M) : 0.f;
        float S = gs[u] * wg;
        S += __shfl_xor_sync(0xffffffffu, S, 8);
        S += __shfl_xor_sync(0xffffffffu, S, 16);
#pragma unroll
        for (int i = 0; i < N; ++i) {
          float x = go[u][i] * wg;
          x += __shfl_xor_sync(0xffffffffu, x, 8);
          x += __shfl_xor_sync(0xffffffffu, x, 16);
          go[u][i] = x;
        }
        m[u] = M;
        l[u] = S;
        const int src = (PL * lane) / N, base = (PL * lane) % N;
#pragma unroll
        for (int jj = 0; jj < N; ++jj) {
          const float x = __shfl_sync(0xffffffffu, go[u][jj], src);
#pragma unroll
          for (int i = 0; i < PL; ++i)
            if (jj == base + i) o[u][i] = x;
        }
      }
    } else {
    // unshared stage
    for (int t0 = 0; t0 < L; t0 += kTok) {
      int slot[kTok];
      KvRaw<DKV, PL> kr[kTok], vr[kTok];
#pragma unroll
      for (int w = 0; w < kTok; ++w) {
        const int t = t0 + w;
        int sl = __shfl_sync(0xffffffffu, my_slot, t & 31);
        if (t >= L) sl = -1;
        else if (t >= 32) {   // rows longer than a warp: read the entry directly
          sl = a.slot_table[((size_t)r * a.W + j) * a.T + t];
          if (sl < 0 || sl >= TW) {
            if (lane == 0) set_status(hdr, BEAMDEC_ERR_DEVICE_CHECK);
            sl = -1;
          }
        }
        slot[w] = sl;
        if (sl >= 0) {
          const size_t e = (((size_t)r * TW + sl) * a.Hkv + g) * D + lane * PL;
          kr[w].load(a.unshared_k, e);
          vr[w].load(a.unshared_v, e);
        }
      }
#pragma unroll
      for (int w = 0; w < kTok; ++w) {
        if (slot[w] < 0) continue;
        float k[PL], v[PL];
        kr[w].to_float(k);
        vr[w].to_float(v);
#pragma unroll
        for (int u = 0; u < kGq; ++u) {
          if (u >= ng) continue;
          float sdot = 0.f;
#pragma unroll
          for (int i = 0; i < PL; ++i) sdot = fmaf(q[u][i], k[i], sdot);
          sdot = warp_sum(sdot);
          const float mn = fmaxf(m[u], sdot);
          const float alpha = ex2(m[u] - mn), pt = ex2(sdot - mn);
          l[u] = l[u] * alpha + pt;
#pragma unroll
          for (int i = 0; i < PL; ++i) o[u][i] = fmaf(pt, v[i], o[u][i] * alpha);
          m[u] = mn;
        }
      }
    }
    }
    // merge with the shared-stage partials of every prompt split
#pragma unroll
    for (int u = 0; u < kGq; ++u) {
      if (u >= ng) continue;
      const size_t row = (size_t)j * G + g0 + u;
      float M = m[u];
      for (int c = 0; c < n_split; ++c) {
        const float mc = c < 32 ? __shfl_sync(0xffffffffu, pm[u], c)
                                : part.m[(((size_t)c * a.R + r) * a.Hkv + g) * rows + row];
        M = fmaxf(M, mc);
      }
      const float wu = (l[u] == 0.f) ? 0.f : ex2(m[u] - M);
      float Lsum = l[u] * wu;
      float O[PL];
#pragma unroll
      for (int i = 0; i < PL; ++i) O[i] = o[u][i] * wu;
      // splits in batches of kBatch whose partial outputs are loaded together
      // (one memory round trip per batch instead of one per split); split 0's
      // output was prefetched with the queries
      // (two with the group stage, whose registers then hold no spill:
      // open-vocabulary step 2436 -> 2351 us)
      constexpr int kBatch = kGrp ? 2 : 8;
      for (int c0 = 0; c0 < n_split; c0 += kBatch) {
        float oc[kBatch][PL];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int c = c0 + k;
          if (c == 0) {
#pragma unroll
            for (int i = 0; i < PL; ++i) oc[k][i] = o0[u][i];
          } else if (c < n_split) {
            const float* src = part.o + ((((size_t)c * a.R + r) * a.Hkv + g) * rows + row) * D + lane * PL;
            if constexpr (PL == 4) {
              const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
              oc[k][0] = x.x; oc[k][1] = x.y; oc[k][2] = x.z; oc[k][3] = x.w;
            } else {
              const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
              oc[k][0] = x.x; oc[k][1] = x.y;
            }
          }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int c = c0 + k;
          if (c >= n_split) break;
          const size_t pi = (((size_t)c * a.R + r) * a.Hkv + g) * rows + row;
          const float mc = c < 32 ? __shfl_sync(0xffffffffu, pm[u], c) : part.m[pi];
          const float lc = c < 32 ? __shfl_sync(0xffffffffu, pl[u], c) : part.l[pi];
          if (lc == 0.f) continue;
          const float w = ex2(mc - M);
          Lsum = fmaf(lc, w, Lsum);
#pragma unroll
          for (int i = 0; i < PL; ++i) O[i] = fmaf(oc[k][i], w, O[i]);
        }
      }
      const float inv = vs / Lsum;
#pragma unroll
      for (int i = 0; i < PL; ++i) O[i] *= inv;
      store_lane<DQ, DKV, D>(a.out, (head0 + g0 + u) * D + lane * PL, O, a.out_dtype);
    }
  }
}

template <int DQ, int DKV, int D>
int launch_t(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream) {
  const int threads = 256;
  const long long warps = (long long)a.R * a.W * a.Hkv;
  dim3 grid((unsigned)((warps + 7) / 8));
  AttnPartials part = attn_partials(a.ws, a.R, a.W, a.Hq, a.Hkv, a.d, p.n_split);
  const auto al16 = [](const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15) == 0; };
  const bool grouped = a.step + 1 >= 8 && al16(a.q) && al16(a.unshared_k) && al16(a.unshared_v);
  prof_begin(kKAttnMerge, stream);
  if (grouped)
    bd_attn_merge_kernel<DQ, DKV, D, true><<<grid, threads, 0, stream>>>(a, p.n_split, part);
  else
    bd_attn_merge_kernel<DQ, DKV, D, false><<<grid, threads, 0, stream>>>(a, p.n_split, part);
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
