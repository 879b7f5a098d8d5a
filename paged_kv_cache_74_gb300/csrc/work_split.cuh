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
__host__ __device__ __forceinline__ long long div_ll(long long a, long long b) {
  if (((a | b) >> 31) == 0) return static_cast<unsigned>(a) / static_cast<unsigned>(b);
  return a / b;
}

// Equal split of W tiles over C CTAs: CTA c owns [range_lo(c), range_lo(c+1)).
__host__ __device__ __forceinline__ long long range_lo(long long W, int C, int c) {
  const long long q = div_ll(W, C), rem = W - q * C;
  return static_cast<long long>(c) * q + (c < rem ? c : rem);
}

// The CTA whose range holds tile t (0 <= t < W).
__host__ __device__ __forceinline__ int cta_of_tile(long long W, int C, long long t) {
  const long long q = div_ll(W, C), rem = W - q * C;
  const long long big = rem * (q + 1);
  if (t < big) return static_cast<int>(div_ll(t, q + 1));
  return static_cast<int>(rem + div_ll(t - big, q));
}

// Lengths the rows of a pa_prefill_varlen batch must keep to (the same
// checks in both of its kernels).
struct RowLimits {
  int max_query_len, max_seq_len, max_tokens, total_q;
};

// A request's prefill rows (q_len > 1 and lengths in range), else ntq = 0.
struct TileReq {
  int q0, q_len, seq_len, ctx, ntq;
};

// From query_start_loc[r], [r + 1] and seq_lens[r] of request r.
__host__ __device__ __forceinline__ TileReq tile_req(int q0, int q1, int seq_len, const RowLimits& l) {
  TileReq p{0, 0, 0, 0, 0};
  const int q_len = q1 - q0;
  if (q_len <= 1) return p;
  if (q_len > seq_len || seq_len > l.max_seq_len || seq_len > l.max_tokens || q_len > l.max_query_len ||
      q0 < 0 || q0 + q_len > l.total_q)
    return p;
  p.q0 = q0;
  p.q_len = q_len;
  p.seq_len = seq_len;
  p.ctx = seq_len - q_len;
  p.ntq = (q_len + 127) / 128;
  return p;
}

// 128-key steps of all 128-row query tiles of a request (one head pair): the
// last tile ends at seq_len, every other one 128 rows before the next.
__host__ __device__ __forceinline__ int tile_req_steps(const TileReq& p) {
  if (p.ntq == 0) return 0;
  return (p.ntq - 1) * p.ntq / 2 + (p.ntq - 1) * ((p.ctx + 127) / 128) + (p.seq_len + 127) / 128;
}

// 16-token tiles (per kv head) of a decode row (q_len == 1, lengths in
// range), else 0.
__host__ __device__ __forceinline__ int decode_row_tiles(int q0, int q1, int seq_len, const RowLimits& l) {
  if (q1 - q0 != 1 || q0 < 0 || q0 >= l.total_q) return 0;
  if (seq_len < 1 || seq_len > l.max_seq_len || seq_len > l.max_tokens) return 0;
  return (seq_len + kBlockSize - 1) / kBlockSize;
}

// Cost of the tile kernel's work: kCostStep per key step, kCostUnit per unit
// (its Q load, first S before any softmax, epilogue).
constexpr long long kCostStep = 4;
constexpr long long kCostUnit = 10;

// SM time (ns on one SM) per unit of tile cost and per 16-token decode tile
// of one kv head, bf16 and e4m3 caches: the weights of the split below.
// From the kernels' own rates on this GPU (a 128 x 128 x 2-head key step
// takes 2.3 us of an SM in long prefill batches, the streaming decode's
// three CTAs of an SM clear a tile every 0.21 us), the tile weight then
// raised to the value that gave the shortest mixed step (583, 700 and 850
// measured: the tile kernel's CTAs start and merge more often in a short
// batch); e4m3 in proportion to the e4m3 kernels' measured times.
constexpr long long kTileNsPerCost = 850;
constexpr long long kDecodeNsPerTile = 211;
constexpr long long kTileNsPerCost8 = 1275;
constexpr long long kDecodeNsPerTile8 = 165;

// Above this tile work per SM (ns) the tile kernel's fixed costs per CTA
// (start-up, merges, the spread of its finish times) are small next to its
// work, and a split of the SMs would only trade them for the error of the
// time model above.
constexpr long long kSplitMaxTileNsPerSm = 150000;

// A pa_prefill_varlen call with both prefill tiles and decode rows: how many
// of the num_sms SMs the tile kernel's CTAs work on, so that its SM time and
// the decode rows' are spread over the SMs in proportion.  The tile CTAs past
// this count exit at once, and the decode CTAs that start on their SMs take
// all the decode rows; the others (started only as tile CTAs finish) find no
// work.  num_sms: no split (every tile CTA works, then the decode rows take
// every SM); 0: no tile work.  Both kernels compute it from the same batch
// sums.
__host__ __device__ __forceinline__ int tile_kernel_sms(long long tile_cost, long long decode_tiles, int num_sms,
                                               bool e4m3) {
  if (tile_cost <= 0) return 0;
  const long long t = tile_cost * (e4m3 ? kTileNsPerCost8 : kTileNsPerCost);
  const long long d = decode_tiles * (e4m3 ? kDecodeNsPerTile8 : kDecodeNsPerTile);
  if (decode_tiles <= 0 || t > kSplitMaxTileNsPerSm * num_sms) return num_sms;
  const long long n = (static_cast<long long>(num_sms) * t + (t + d) / 2) / (t + d);
  return static_cast<int>(n < 1 ? 1 : (n > num_sms ? num_sms : n));
}

// CTAs of a decode grid of num_ctas (ctas_per_sm on each of num_sms SMs)
// that take the decode rows when the tile kernel keeps tile_sms SMs.
__host__ __device__ __forceinline__ int decode_split_ctas(int tile_sms, int num_sms, int num_ctas, int ctas_per_sm) {
  if (tile_sms <= 0 || tile_sms >= num_sms) return num_ctas;
  return num_ctas - ctas_per_sm * tile_sms;
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
