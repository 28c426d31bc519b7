// Shared device helpers of libbeamdec (CUDA side only).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/beamdec.h"

namespace bd {

constexpr int kWsHeaderBytes = 256;   // status word, grid-barrier counters

// First 256 bytes of every compute workspace.
struct WsHeader {
  int32_t status;        // first device-detected error (BEAMDEC_ERR_*), 0 = clean
  uint32_t bar_count;    // grid barrier arrivals (returns to 0 after each barrier)
  uint32_t bar_gen;      // grid barrier generation
  // Test hooks of the bounded waits, written by the caller (0 in normal use;
  // the zero-filled workspace starts that way and the library never sets
  // them): poll_limit replaces the grid barrier's default poll count;
  // bar_extra adds arrivals that no block ever supplies to the grid barrier,
  // so each of its waits runs out and reports BEAMDEC_ERR_TIMEOUT;
  // probe_polls makes each CTA of the tensor-core kernels (attention shared
  // stage, LM head) first wait that many polls on an mbarrier that nothing
  // completes, before it issues any copy or MMA, so the wait runs out and
  // the CTA takes its timeout exit.
  uint32_t poll_limit;
  uint32_t bar_extra;
  uint32_t probe_polls;
  // attention workspaces: the prompt K/V (and its row count) whose bf16 copy
  // the workspace holds, written by the dequantisation kernel
  unsigned long long prep_k, prep_v, prep_rows, prep_dst;
  uint32_t pad[50];
};
static_assert(sizeof(WsHeader) == kWsHeaderBytes, "header size");

__device__ __forceinline__ void set_status(WsHeader* h, int code) {
  atomicCAS(&h->status, 0, code);
}

// ---- order-preserving float keys ------------------------------------------
// desc_key(s): smaller key <=> larger s; -0 and +0 map to one key.
__device__ __forceinline__ uint32_t desc_key(float s) {
  uint32_t b = __float_as_uint(s);
  if (b == 0x80000000u) b = 0u;
  uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ~ord;
}
__device__ __forceinline__ float desc_key_value(uint32_t k) {
  uint32_t ord = ~k;
  uint32_t b = (ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord;
  return __uint_as_float(b);
}

// Global pool key: desc(score) << 32 | beam << 18 | index, where index is the
// candidate's position among its beam's candidates (the child position within
// the trie node, whose codes ascend, or the token itself with no trie).  Within
// one beam the index order is the token order, so ascending keys order
// candidates by (score desc, beam asc, token asc).
constexpr int kTokBits = 18;
constexpr int kBeamBits = 13;
__device__ __forceinline__ uint64_t pool_key(uint32_t k32, int beam, int tok) {
  return ((uint64_t)k32 << 32) | ((uint64_t)beam << kTokBits) | (uint64_t)tok;
}
__device__ __forceinline__ int pool_key_beam(uint64_t k) {
  return (int)((k >> kTokBits) & ((1u << kBeamBits) - 1));
}
__device__ __forceinline__ int pool_key_tok(uint64_t k) { return (int)(k & ((1u << kTokBits) - 1)); }

// ---- fast base-2 exponential (the hardware instruction) -------------------
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// ---- warp / block reductions ----------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---- bounded grid barrier (cooperative launches only) ---------------------
// Every block of the grid must call it the same number of times.  The wait is
// bounded: after `limit` polls the block records BEAMDEC_ERR_TIMEOUT and goes
// on, so a broken launch ends with an error instead of a hung GPU.
__device__ __forceinline__ void grid_barrier(WsHeader* h, unsigned nblocks) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t hook = *reinterpret_cast<volatile uint32_t*>(&h->poll_limit);
    const long long limit = hook ? (long long)hook : (1ll << 26);
    const uint32_t target = nblocks + *reinterpret_cast<volatile uint32_t*>(&h->bar_extra);
    volatile uint32_t* gen = &h->bar_gen;
    uint32_t g = *gen;
    __threadfence();
    uint32_t arrived = atomicAdd(&h->bar_count, 1u) + 1u;
    if (arrived == target) {
      atomicExch(&h->bar_count, 0u);
      __threadfence();
      atomicAdd(&h->bar_gen, 1u);
    } else {
      long long it = 0;
      while (*gen == g) {
        if (++it > limit) { set_status(h, BEAMDEC_ERR_TIMEOUT); break; }
        __nanosleep(64);
      }
    }
    __threadfence();
  }
  __syncthreads();
}

}  // namespace bd
