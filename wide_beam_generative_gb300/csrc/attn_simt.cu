// Shared stage of the beam attention on CUDA cores (fp32 FMA).
//
// "Generative recommendation design" (xLLM) §4.2.1-§4.2.2: the prompt KV is
// stored once per request and every beam attends to it; the shared stage
// produces, per query row, the partial softmax statistics and output over the
// prompt only.  A query row is (beam j, query head h) of one kv head g: the
// W*G rows of (request, g) all read the same prompt keys, so a block stages a
// 32-key tile of K and V once in shared memory for 32 rows.
//
// This kernel serves fp32 workloads (and any shape the tensor-core kernel
// does not take).  Layout per thread: 4 threads per query row, thread p owns
// the dims {16i + 4p .. 16i + 4p + 3}, so the 4 threads of a row read
// consecutive 16-byte words of a staged key (no bank conflicts).
#include <cuda_runtime.h>
#include <math.h>

#include "attn_common.cuh"
#include "common.cuh"
#include "internal.h"

namespace bd {
namespace {

constexpr int kRows = 32;
constexpr int kKeys = 32;

template <int DQ, int DKV, int D>
__global__ void __launch_bounds__(128)
bd_attn_shared_simt_kernel(AttnArgs a, int n_split, int split_len, AttnPartials part) {
  __shared__ __align__(16) float Ks[kKeys][D];
  __shared__ __align__(16) float Vs[kKeys][D];
  const int tile = blockIdx.x;
  const int g = blockIdx.y % a.Hkv;
  const int sp = blockIdx.y / a.Hkv;
  const int r = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  const int rows = a.W * G;
  const int row0 = tile * kRows;
  if (row0 >= a.n_live[r] * G) return;   // every row of the tile is a dead beam
  const int tid = threadIdx.x, lr = tid >> 2, p = tid & 3;
  const int row = row0 + lr;
  const bool valid = row < rows;
  const int j = valid ? row / G : 0, gi = valid ? row - (row / G) * G : 0;
  const int pbase = a.prompt_offsets[r];
  const int P = a.prompt_offsets[r + 1] - pbase;
  const int k0 = sp * split_len;
  const int k1 = min(P, k0 + split_len);
  constexpr int NQ = D / 16;
  const float ks = (DKV == 2 && a.k_scale) ? a.k_scale[g] : 1.f;
  const float scale2 = a.sm_scale * kLog2e * ks;
  float4 q[NQ], o[NQ];
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid)
      v = load4<DQ>(a.q, (((size_t)r * a.W + j) * a.Hq + g * G + gi) * D + i * 16 + p * 4);
    q[i] = make_float4(v.x * scale2, v.y * scale2, v.z * scale2, v.w * scale2);
    o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY, l = 0.f;
  for (int kb = k0; kb < k1; kb += kKeys) {
    const int nk = min(kKeys, k1 - kb);
    __syncthreads();
    for (int idx = threadIdx.x; idx < kKeys * D / 4; idx += 128) {
      const int kk = idx / (D / 4), c = (idx - kk * (D / 4)) * 4;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (kk < nk) {
        const size_t e = ((size_t)(pbase + kb + kk) * a.Hkv + g) * D + c;
        kv = load4<DKV>(a.shared_k, e);
        vv = load4<DKV>(a.shared_v, e);
      }
      *reinterpret_cast<float4*>(&Ks[kk][c]) = kv;
      *reinterpret_cast<float4*>(&Vs[kk][c]) = vv;
    }
    __syncthreads();
    for (int kk = 0; kk < nk; kk += 8) {
      float s[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          const float4 kx = *reinterpret_cast<const float4*>(&Ks[kk + u][i * 16 + p * 4]);
          acc = fmaf(q[i].x, kx.x, acc);
          acc = fmaf(q[i].y, kx.y, acc);
          acc = fmaf(q[i].z, kx.z, acc);
          acc = fmaf(q[i].w, kx.w, acc);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        s[u] = (kk + u < nk) ? acc : -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int u = 1; u < 8; ++u) mx = fmaxf(mx, s[u]);
      const float mn = fmaxf(m, mx);
      const float alpha = ex2(m - mn);
      l *= alpha;
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        o[i].x *= alpha; o[i].y *= alpha; o[i].z *= alpha; o[i].w *= alpha;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float pu = ex2(s[u] - mn);
        l += pu;
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          const float4 vx = *reinterpret_cast<const float4*>(&Vs[kk + u][i * 16 + p * 4]);
          o[i].x = fmaf(pu, vx.x, o[i].x);
          o[i].y = fmaf(pu, vx.y, o[i].y);
          o[i].z = fmaf(pu, vx.z, o[i].z);
          o[i].w = fmaf(pu, vx.w, o[i].w);
        }
      }
      m = mn;
    }
  }
  if (!valid) return;
  const size_t pi = (((size_t)sp * a.R + r) * a.Hkv + g) * rows + row;
  if (p == 0) { part.m[pi] = m; part.l[pi] = l; }
#pragma unroll
  for (int i = 0; i < NQ; ++i)
    *reinterpret_cast<float4*>(part.o + pi * D + i * 16 + p * 4) = o[i];
}

template <int DQ, int DKV, int D>
int launch_t(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  dim3 grid((a.W * G + kRows - 1) / kRows, a.Hkv * p.n_split, a.R);
  AttnPartials part = attn_partials(a.ws, a.R, a.W, a.Hq, a.Hkv, a.d, p.n_split);
  prof_begin(kKAttnSimt, stream);
  bd_attn_shared_simt_kernel<DQ, DKV, D><<<grid, 128, 0, stream>>>(a, p.n_split, p.split_len, part);
  prof_end(kKAttnSimt, stream);
  return cudaGetLastError() == cudaSuccess ? BEAMDEC_OK : BEAMDEC_ERR_CUDA;
}

}  // namespace

int launch_attn_shared_simt(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream) {
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
