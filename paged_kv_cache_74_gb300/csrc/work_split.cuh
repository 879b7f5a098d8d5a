// work_split.cuh -- the equal split of a batch's numbered work steps over
// the CTAs of a persistent grid, and the epoch-tagged counter that picks
// the last contributor of a piece of work shared by several CTAs (it merges
// the pieces: "vLLM 深度解析（二）：PagedAttention 核心机制", sections 3.2.7
// and 3.3).  Used by the decode kernels and the prefill kernel.
#pragma once

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

// 64-bit division, through 32-bit unsigned division when both operands fit
// (a 64-bit division is a long instruction sequence).
__device__ __forceinline__ long long div_ll(long long a, long long b) {
  if (((a | b) >> 31) == 0) return static_cast<unsigned>(a) / static_cast<unsigned>(b);
  return a / b;
}

// Equal split of W tiles over C CTAs: CTA c owns [range_lo(c), range_lo(c+1)).
__device__ __forceinline__ long long range_lo(long long W, int C, int c) {
  const long long q = div_ll(W, C), rem = W - q * C;
  return static_cast<long long>(c) * q + (c < rem ? c : rem);
}

// The CTA whose range holds tile t (0 <= t < W).
__device__ __forceinline__ int cta_of_tile(long long W, int C, long long t) {
  const long long q = div_ll(W, C), rem = W - q * C;
  const long long big = rem * (q + 1);
  if (t < big) return static_cast<int>(div_ll(t, q + 1));
  return static_cast<int>(rem + div_ll(t - big, q));
}

// The last contributor of a pair clears its counter once it has merged:
// every launch then leaves the counters at zero, so a launch replayed with
// the same epoch (a CUDA graph) starts from clean counters too.
__device__ __forceinline__ void release_pair(unsigned long long* counter) {
  atomicExch(counter, 0ull);
}

// Registers this CTA's partial for a pair; true if it was the last of n.
// The first exchange assumes the other n - 1 have already counted (no read
// before it): the contributor that finishes a pair pays one round trip.
__device__ bool contribute(unsigned long long* counter, unsigned epoch, int n, int32_t* status,
                           int who) {
  unsigned long long old = (static_cast<unsigned long long>(epoch) << 32) |
                           static_cast<unsigned>(n > 1 ? n - 1 : 0);
  unsigned long long now = 0;
  for (int tries = 0; tries < (1 << 20); ++tries) {
    now = (static_cast<unsigned>(old >> 32) == epoch)
              ? old + 1
              : ((static_cast<unsigned long long>(epoch) << 32) | 1ull);
    const unsigned long long seen = atomicCAS(counter, old, now);
    if (seen == old) return static_cast<int>(now & 0xffffffffu) == n;
    old = seen;
  }
  record_error(status, PA_DEV_WAIT_TIMEOUT, who, 3);
  return false;
}

}  // namespace
}  // namespace pa
