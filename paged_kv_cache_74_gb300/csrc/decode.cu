// decode.cu -- paged decode attention for sm_103a.
//
// Method ("vLLM 深度解析（二）：PagedAttention 核心机制"):
//   section 3.1  a request's token t lives in physical block
//                block_table[r][t / 16] at offset t % 16;
//   section 2.2  online softmax: a running (m, l, A) per query row, merged
//                tile by tile, O = A / l at the end;
//   section 3.2  masked scores of tokens >= seq_len are excluded and the V
//                of out-of-context slots is zeroed before it is used;
//   sections 3.2.7, 3.2.9, 3.3  a long context is cut into pieces whose
//                (m_j, l_j, O_j) are merged: m = max m_j,
//                L = sum l_j e^{m_j - m}, O = sum O_j l_j e^{m_j - m} / L.
//
// GB300 design.  Decode is HBM-bound, so the kernel is built around keeping
// HBM busy; the products are small and must not hold the K/V stages long:
//
// * Balanced persistent grid.  Every (request, kv head, 16-token block)
//   tile of the batch is numbered (request-major, then kv head, then block)
//   and the W tiles are cut into equal contiguous ranges, one per CTA, with
//   as many CTAs as fit on the GPU at once.  No CTA idles at the tail and
//   the K/V stream of a CTA never drains between requests.  A range covers
//   whole (request, kv head) pairs, written straight to `out`, and at most
//   two pieces of pairs shared with the neighbouring ranges; those are
//   written as partials (m_j, l_j, O_j) and merged by the contributor that
//   finishes last (an epoch-tagged counter per pair decides which).  Behind
//   a small prefill tile batch of the same pa_prefill_varlen call
//   (`tile_sms`), the ranges go only to the CTAs that start on the SMs the
//   tile kernel leaves (tile_kernel_sms()); the rest find no work.
// * One CTA serves every q head of a kv head, so each K/V byte is read from
//   HBM once.  A producer warp reads block ids 32 at a time and issues one
//   TMA tensor load per (block, kv head) tile of K and of V (16 tokens x
//   head_dim, 4 KB at head_dim 128 in bf16) into an 8-stage ring (16
//   stages of the half-size e4m3 tiles; at head_dim 128 with 4 q heads per
//   kv head an e4m3 unit is two kv heads, 8 q heads, whose tiles come in
//   one 4 KB copy: copies of 2 KB stream at about half the bytes per
//   second of 4 KB ones at the same bytes in flight) guarded by mbarriers, writes each stage's block index and flags next to it, and
//   prefetches each segment's q with a bulk copy into a double buffer.
// * Two consumer warps take alternate stages.  A warp computes S^T = K q^T
//   (16 tokens x 8 columns of q heads, padding heads zero) and
//   O^T += V^T P^T with warp-level m16n8k16 tensor-core products: K and V
//   fragments come straight from the stage with ldmatrix (the copies land
//   swizzled, so those reads are conflict-free), the weights P go from the
//   score fragments to the operand fragments with movmatrix.  A tile costs
//   about 0.5 us, so the stage is released soon after it lands.  bf16
//   caches: bf16 products, P rounded to bf16.  e4m3 caches (KV8): the K
//   and V bytes are converted to f16 in registers (exact: every e4m3 value
//   is an f16 value), q and P are rounded to f16, and the head_dim order of
//   the fragments follows the bytes ldmatrix delivers (see below).  l sums
//   the rounded weights.  At a segment end the two warps merge their
//   states through shared memory and hand the result to an epilogue warp,
//   which writes the output or the partial, bumps the pair counter and, as
//   last contributor, merges the partials; the consumers go straight on to
//   the next segment.
// * The running max is rescaled lazily, only when a new score exceeds the
//   reference by more than 2^8 (O = A / l is exact for any reference), and
//   each segment is padded to a multiple of the consumer count in stages,
//   so both consumers finish it together.
// * The x-split layout of section 3.2.1 (XS) runs through the bf16 path with
//   other TMA views: K as 8-token x 16-byte rows (128-byte swizzled), V as
//   V^T [head_dim][16 tokens] (32-byte swizzled), which is already the
//   operand layout of O^T += V^T P^T.
#include "decode_common.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr float kNegBig = -1e30f;      // finite stand-in for -inf in running maxima

// Order-preserving unsigned keys of floats (no NaN): larger float, larger key.
__device__ __forceinline__ unsigned float_to_max_key(float f) {
  const unsigned b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float max_key_to_float(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
constexpr float kRescaleSlack = 8.0f;  // log2 units

// Stage flags (written by the producer next to each ring stage).
constexpr int kSkip = 1;     // padding stage: no data, nothing to compute
constexpr int kLastRow = 2;  // the segment ends after this row of stages
constexpr int kDone = 4;     // no more work for the warp that receives it
constexpr int kEndSeg = 3;   // segment kind handed to the epilogue warp: no more segments


template <int D, int GMAX, bool KV8 = false, bool XS = false>
struct DecodeCfg {
  // Two consumer warps take alternate stages; each computes q.k and p.v of
  // a 16-token tile as warp-level m16n8k16 tensor-core products (tokens /
  // head_dim x 8 padded q heads), bf16 for bf16 caches, f16 for e4m3 ones.
  // One 16-token tile takes ~0.5 us, so two warps keep up with the stream.
  static constexpr int NC = 2;
  static constexpr int MINB = 3;                               // CTAs per SM
  static constexpr int ELT = KV8 ? 1 : 2;                      // bytes per K/V element (e4m3 / bf16)
  static constexpr int KS = D / 16;                            // 16-wide steps of head_dim
  // e4m3 units of two kv heads (8 q heads: GMAX 8): a tile holds both
  // heads' 16 tokens, [token][kv head][head_dim] bytes, one copy for both.
  static constexpr bool PAIR = KV8 && !XS && GMAX == 8;
  static constexpr int TILE = kBlockSize * D * ELT * (PAIR ? 2 : 1);  // bytes of one K (or V) tile
  // A multiple of NC (see below).  Plain e4m3 tiles are half as large:
  // twice as many fit, and the same bytes are in flight.
  static constexpr int STAGES = (D == 128 ? 8 : 16) * (KV8 && !PAIR ? 2 : 1);
  // shared memory carve-up (bytes)
  static constexpr int RING = STAGES * 2 * TILE;
  // The consumers hand every finished segment to an epilogue warp (partial
  // write, pair counter, last-contributor merge), so the global round trips
  // of a segment end never stall the K/V stream.
  static constexpr int WF = GMAX * D + 2 * GMAX;               // floats of one (O, m, l) record
  static constexpr int HF = WF + 8;                            // ... plus the segment record
  static constexpr int HAND = (HF * 4 + 15) / 16 * 16;         // the segment handed over
  static constexpr int QBUF = 2 * GMAX * D * 2;                // q of two segments
  static constexpr int OFF_HAND = RING;
  static constexpr int OFF_Q = OFF_HAND + HAND;
  static constexpr int OFF_META = OFF_Q + QBUF;                // int2 per stage
  static constexpr int OFF_SEG = OFF_META + STAGES * 8;        // 2 segment records
  static constexpr int OFF_BAR = OFF_SEG + 2 * 32;  // full, empty, qfull, qempty, sync, hfull, hempty
  static constexpr int OFF_MISC = OFF_BAR + (2 * STAGES + 7) * 8;
  static constexpr int SMEM = OFF_MISC + 32;
  static constexpr int THREADS = (NC + 2) * 32;                // + producer and epilogue warps
  // Stage i goes to consumer warp i % NC.  With STAGES a multiple of NC a
  // stage is only ever used by one warp, so when a warp waits on a stage
  // the barrier is at most one phase behind and the parity wait is exact.
  static_assert(STAGES % NC == 0, "each ring stage must belong to one consumer warp");
  static_assert(SMEM <= 227 * 1024 && MINB * (SMEM + 1024) <= 228 * 1024,
                "shared memory must allow MINB CTAs per SM");
  static_assert(GMAX <= 8 && NC == 2, "an m16n8k16 product serves at most 8 q heads");
  static_assert(!PAIR || D == 128, "two-head e4m3 tiles: head_dim 128 (128-byte rows)");
  // Bulk-copy destinations (ring, q) 16-byte aligned; the segment records'
  // 64-bit fields 8-byte aligned.
  static_assert(RING % 1024 == 0 && OFF_HAND % 16 == 0 && OFF_Q % 16 == 0 && OFF_META % 8 == 0 &&
                    OFF_SEG % 8 == 0 && OFF_BAR % 8 == 0 && OFF_MISC % 8 == 0 && (WF * 4) % 8 == 0,
                "shared-memory carve-up alignment");
  static_assert(GMAX * D / 2 % 32 == 0, "the epilogue lanes split the head_dim pairs evenly");
};

// What the producer tells the consumers about a segment: the run of blocks
// of one (request, kv head) pair inside this CTA's range.
struct SegInfo {
  int row;        // q / out row of the request
  int seq_len;
  int nblk;       // blocks of the request
  int kind;       // kWhole, kHead or kTail
  long long t0;   // number of the pair's first tile
  int r;
  int kvh;
};
static_assert(sizeof(SegInfo) <= 32, "segment record");

// ---- x-split layout ("vLLM 深度解析（二）：PagedAttention 核心机制", section
// 3.2.1): K [blocks, kv heads, head_dim / 8, block, 8] (8 bf16 = 16 bytes
// innermost), V [blocks, kv heads, head_dim, block].
//
// A K stage holds one 16-token tile as [head_dim / 8 chunks][2 token groups]
// [8 tokens x 16 bytes]: 128-byte rows r = 2 c + t / 8, the 16-byte unit of
// token t at (t % 8) ^ (r % 8) (the copy's 128-byte swizzle).  Lanes reading
// chunk c of one token then hit distinct bank groups.
__device__ __forceinline__ uint32_t xs_k_offset(int t, int c) {
  const int r = 2 * c + (t >> 3);
  return static_cast<uint32_t>(r * 128 + (((t & 7) ^ (r & 7)) * 16));
}

// A V stage of the x-split layout holds V^T of the tile as [head_dim][16
// tokens]: 32-byte rows, the two 16-byte halves (tokens 0-7, 8-15) swapped
// on rows with bit 2 set (the copy's 32-byte swizzle).  Offset of half tb
// of row d:
__device__ __forceinline__ uint32_t xs_v_offset(int d, int tb) {
  return static_cast<uint32_t>(d * 32 + ((tb ^ ((d >> 2) & 1)) * 16));
}

// e4m3 x-split stages: K as [head_dim / 16 chunks][16 tokens][16 B], V as
// V^T [head_dim][16 tokens] (bytes, no swizzle: 8 consecutive 16-byte rows
// are conflict-free).  A plain ldmatrix of V^T gives a lane tokens 4 ft ..
// 4 ft + 3 of its head_dim row, so the products' token order is permuted:
// product row r of S (and index r of the P.V reduction) is token xs8_token(r),
// i.e. rows 2 t, 2 t + 1 are tokens 4 t, 4 t + 1 and rows 2 t + 8, 2 t + 9
// are tokens 4 t + 2, 4 t + 3.  The K rows are read in that order.
__device__ __forceinline__ int xs8_token(int r) {
  return r < 8 ? 4 * (r >> 1) + (r & 1) : 4 * ((r - 8) >> 1) + 2 + (r & 1);
}

// A token-major K or V stage (the grouped copy, 128-byte swizzled):
// [8-token group][head_dim / 64][8 tokens][128 B], the 16-byte chunk c of
// token t at unit (c % 8) ^ (t % 8) of its 128-byte row.
template <int D>
__device__ __forceinline__ uint32_t grp_offset(int t, int c) {
  return static_cast<uint32_t>((t >> 3) * (D / 64) * 1024 + (c >> 3) * 1024 + (t & 7) * 128 +
                               (((c & 7) ^ (t & 7)) * 16));
}

// ---- warp-level tensor-core helpers (m16n8k16, bf16 in, fp32 accumulate)
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// d += A (16 x 16, row-major fragments a) * B (16 x 8, column fragments b0, b1).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// The transpose of an 8 x 8 bf16 matrix held one row pair per lane.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// ---- e4m3 caches on the tensor cores (f16 products, fp32 accumulate).
// Every e4m3 value is exact in f16, so K and V lose nothing in the
// conversion; q and the weights are rounded to f16 (|q| saturates at 65504).
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Two e4m3 values (low byte first) as f16x2 (low half first).
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(two)));
  return h2;
}
// Bytes (b0, b2, b1, b3) of x.
__device__ __forceinline__ uint32_t bytes_0213(uint32_t x) {
  uint32_t y;
  asm("prmt.b32 %0, %1, 0, 0x3120;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
  uint32_t h2;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(h2) : "f"(hi), "f"(lo));
  return h2;
}
__device__ __forceinline__ float f16_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
// A K or V stage of an e4m3 cache: [16 tokens][head_dim bytes] through a
// swizzled copy (128-byte rows: 16-byte chunk c of token t at c ^ (t % 8);
// 64-byte rows: at c ^ ((t / 2) % 4)), so ldmatrix rows of 8 tokens hit 8
// distinct bank groups.
template <int D>
__device__ __forceinline__ uint32_t e8_offset(int t, int c) {
  const int sw = D == 128 ? (t & 7) : ((t >> 1) & 3);
  return static_cast<uint32_t>(t * D + ((c ^ sw) * 16));
}

// Byte offset of 16-byte chunk c of row r of a 128-byte-swizzled tile of
// 128-byte rows (a two-head e4m3 tile: row 2 t + h is token t of head h).
__device__ __forceinline__ uint32_t e8_row_offset(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) * 16));
}

// MIX: the decode rows of a pa_prefill_varlen call that may split the SMs
// with its tile kernel (DecodeArgs::tile_sms); a separate instantiation, so
// that the plain decode's start-up stays as short as it is.
template <int D, int GMAX, bool KV8, bool XS, bool MIX>
__global__ void __launch_bounds__(DecodeCfg<D, GMAX, KV8, XS>::THREADS,
                                  DecodeCfg<D, GMAX, KV8, XS>::MINB)
paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  using C = DecodeCfg<D, GMAX, KV8, XS>;
  const int cta = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  extern __shared__ __align__(1024) uint8_t smem[];
  int2* meta = reinterpret_cast<int2*>(smem + C::OFF_META);
  SegInfo* seginfo = reinterpret_cast<SegInfo*>(smem + C::OFF_SEG);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
  long long* total_tiles = reinterpret_cast<long long*>(smem + C::OFF_MISC + 8);
  int* split_ctas = reinterpret_cast<int*>(smem + C::OFF_MISC + 16);  // CTAs the tiles are split over
  const uint32_t ring_s = smem_u32(smem);
  const uint32_t full0 = smem_u32(smem + C::OFF_BAR);
  const uint32_t empty0 = full0 + 8 * C::STAGES;
  const uint32_t qfull0 = empty0 + 8 * C::STAGES;
  const uint32_t qempty0 = qfull0 + 16;
  const uint32_t csync_bar = qempty0 + 16;  // consumer-warp barrier (bounded waits)
  const uint32_t hfull0 = csync_bar + 8;     // segment handed to the epilogue warp
  const uint32_t hempty0 = hfull0 + 8;       // ... and taken by it
  const uint32_t qbuf_s = smem_u32(smem + C::OFF_Q);

  // TMA destinations must be 128-byte aligned (1024 for the 128-byte
  // swizzled boxes of the bf16 paths); the dynamic shared-memory base always
  // is on this GPU, but never issue a copy if it were not.
  if (ring_s & 1023) {
    griddep_wait();
    if (threadIdx.x == 0) record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, 6);
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(qfull0 + 8 * k, 1);
      mbar_init(qempty0 + 8 * k, C::NC);
    }
    mbar_init(csync_bar, C::NC);
    mbar_init(hfull0, 1);
    mbar_init(hempty0, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (!a.defer_griddep) griddep_wait();  // the cache write before this launch may still be finishing

  if (warp == C::NC) {
    // ================================================================ producer
    if (cta == 0) report_bad_rows(a, lane);
    // Total tiles W of the batch.
    long long nb_sum = 0;
    for (int r = lane; r < a.num_seqs; r += 32) {
      int len, row;
      nb_sum += request_blocks(a, r, &len, &row);
    }
    const long long W = warp_sum_ll(nb_sum) * a.num_kv_heads;
    long long lo, hi;
    if constexpr (MIX) {
      // The tile kernel's cost (the call's prefill rows) sets how many CTAs
      // take the decode rows.
      long long tc_sum = 0;
      for (int r = lane; r < a.num_seqs; r += 32) {
        const TileReq p = tile_req(a.query_start_loc[r], a.query_start_loc[r + 1], a.seq_lens[r], row_limits(a));
        tc_sum += kCostStep * tile_req_steps(p) + kCostUnit * p.ntq;
      }
      const long long Ct = warp_sum_ll(tc_sum) * a.num_kv_heads * ((a.group + 1) / 2);
      const int nct =
          decode_split_ctas(tile_kernel_sms(Ct, W, a.tile_sms, KV8), a.tile_sms, a.num_ctas, a.ctas_per_sm);
      lo = W > 0 && cta < nct ? range_lo(W, nct, cta) : 0;
      hi = W > 0 && cta < nct ? range_lo(W, nct, cta + 1) : 0;
      if (lane == 0) *split_ctas = nct;
    } else {
      lo = W > 0 ? range_lo(W, a.num_ctas, cta) : 0;
      hi = W > 0 ? range_lo(W, a.num_ctas, cta + 1) : 0;
    }
    if (lane == 0) *total_tiles = W;

    int pos = 0;  // stage sequence number
    auto stage_begin = [&](int p) -> bool {  // lane 0: wait until stage p may be refilled
      if (p >= C::STAGES && !mbar_wait(empty0 + 8 * (p % C::STAGES), ((p / C::STAGES) - 1) & 1)) {
        record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, 1);
        *abort_flag = 1;
      }
      return *abort_flag == 0;
    };

    if (lo < hi) {
      // Request holding tile `lo`: scan the per-request tile counts 32 at a time.
      long long base = 0;  // tiles before request r0
      int r0 = -1;
      for (int rc = 0; rc < a.num_seqs && r0 < 0; rc += 32) {
        const int r = rc + lane;
        int len, row;
        const long long nt = r < a.num_seqs ? static_cast<long long>(request_blocks(a, r, &len, &row)) *
                                                  a.num_kv_heads
                                            : 0;
        const long long chunk = warp_sum_ll(nt);
        if (base + chunk <= lo) {  // tile `lo` lies past these 32 requests
          base += chunk;
          continue;
        }
        long long incl = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, r < a.num_seqs && base + incl > lo);
        if (hit) {
          const int first = __ffs(hit) - 1;
          const long long excl = __shfl_sync(0xffffffffu, incl - nt, first);
          r0 = rc + first;
          base += excl;
        } else {
          base += __shfl_sync(0xffffffffu, incl, 31);
        }
      }
      // Block ids: lane L keeps ids 32m + L (m < kRowCache) of the current
      // request and of the next one in registers, so the kv heads of one
      // request and the switch to the next request need no global load on
      // the issue path; ids past the cached ones are fetched one 32-tile
      // chunk ahead.  The next request's length and q range are read early.
      constexpr int kRowCache = 4;
      int cur_ids[kRowCache], nxt_ids[kRowCache];
      int nxt_r = -1, nxt_len = 0, nxt_q0 = 0, nxt_q1 = 0;
      auto load_row = [&](int rr, int (&ids)[kRowCache]) {
        const int32_t* rp = a.block_tables + static_cast<size_t>(rr) * a.max_blocks_per_seq;
#pragma unroll
        for (int m = 0; m < kRowCache; ++m) {
          const int gi = 32 * m + lane;  // tile index
          ids[m] = (rr < a.num_seqs && (gi >> a.tile_shift) < a.max_blocks_per_seq)
                       ? __ldg(rp + (gi >> a.tile_shift))
                       : 0;
        }
      };
      auto prefetch_next = [&](int rr) {
        nxt_r = rr + 1;
        if (nxt_r < a.num_seqs) {
          nxt_len = __ldg(a.seq_lens + nxt_r);
          if (a.query_start_loc != nullptr) {
            nxt_q0 = __ldg(a.query_start_loc + nxt_r);
            nxt_q1 = __ldg(a.query_start_loc + nxt_r + 1);
          }
        }
        load_row(nxt_r, nxt_ids);
      };
      int r = r0, len = 0, row = 0;
      load_row(r, cur_ids);
      int nb = request_blocks(a, r, &len, &row);
      prefetch_next(r);
      long long off = lo - base;
      int kvh = static_cast<int>(off / nb);
      int b = static_cast<int>(off % nb);
      long long t = lo;
      const uint64_t policy = l2_policy_evict_first();
      if (lane == 0) {
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
      }
      int seg = 0;
      bool ok = true;
      while (t < hi && ok) {
        const int seg_n = static_cast<int>(min(hi - t, static_cast<long long>(nb - b)));
        const int kind = (b == 0 && seg_n == nb) ? kWhole : (b > 0 ? kHead : kTail);
        const int slot = seg & 1;
        if (lane == 0) {
          // q and the segment record go to slot seg % 2 once every consumer
          // warp has taken segment seg - 2 from it.
          if (seg >= 2 && !mbar_wait(qempty0 + 8 * slot, ((seg >> 1) - 1) & 1)) {
            record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, 4);
            *abort_flag = 1;
          }
          if (*abort_flag == 0) {
            SegInfo si;
            si.row = row;
            si.seq_len = len;
            si.nblk = nb;
            si.kind = kind;
            si.t0 = base + static_cast<long long>(kvh) * nb;
            si.r = r;
            si.kvh = kvh;
            seginfo[slot] = si;
            const uint32_t qbytes = a.group * D * 2;
            mbar_arrive_expect_tx(qfull0 + 8 * slot, qbytes);
            bulk_copy_g2s(qbuf_s + slot * (GMAX * D * 2),
                          a.q + (static_cast<size_t>(row) * a.num_heads +
                                 static_cast<size_t>(kvh) * a.group) * D,
                          qbytes, qfull0 + 8 * slot);
          }
        }
        ok = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
        const int rows = (seg_n + C::NC - 1) / C::NC;
        const int32_t* rowp = a.block_tables + static_cast<size_t>(r) * a.max_blocks_per_seq;
        const int seg_end = b + seg_n;  // one past the segment's last tile
        int my_id = 0, far_next = 0;
        for (int j = 0; j < rows * C::NC && ok; ++j) {
          if ((j & 31) == 0) {
            const int gi = b + j + lane;  // this lane's tile in the chunk
            int cached = 0;
#pragma unroll
            for (int m = 0; m < kRowCache; ++m) {
              const int v = __shfl_sync(0xffffffffu, cur_ids[m], gi & 31);
              if ((gi >> 5) == m) cached = v;
            }
            if (gi < 32 * kRowCache)
              my_id = cached;
            else if (j == 0)
              my_id = gi < seg_end ? __ldg(rowp + (gi >> a.tile_shift)) : 0;
            else
              my_id = far_next;
            const int gn = gi + 32;  // next chunk, fetched now
            far_next = (gn >= 32 * kRowCache && gn < seg_end) ? __ldg(rowp + (gn >> a.tile_shift)) : 0;
          }
          const int phys = __shfl_sync(0xffffffffu, my_id, j & 31);
          if (lane == 0 && stage_begin(pos)) {
            const int s = pos % C::STAGES;
            const bool real = j < seg_n;
            const int flags = (real ? 0 : kSkip) | (j >= (rows - 1) * C::NC ? kLastRow : 0);
            meta[s] = make_int2(b + j, flags);
            const uint32_t full = full0 + 8 * s;
            if (real) {
              const bool bad = static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks);
              if (bad) record_error(a.status, PA_DEV_BAD_BLOCK_ID, r, phys);
              mbar_arrive_expect_tx(full, 2 * C::TILE);
              if constexpr (XS) {
                // Block coordinate num_blocks is wholly out of bounds: TMA fills zeros.
                const int blk = bad ? a.num_blocks : phys;
                const int sub = (b + j) & ((1 << a.tile_shift) - 1);  // 16-token tile of the block
                const int kvc = kvh / a.kv_div;                        // kv head of the cache
                if constexpr (KV8)  // one contiguous run per chunk: {B x 16 bytes, d / 16, ...}
                  tma_load_4d(ring_s + (2 * s) * C::TILE, &kmap, full, 256 * sub, 0, kvc, blk, policy);
                else
                  tma_load_5d(ring_s + (2 * s) * C::TILE, &kmap, full, 0, 2 * sub, 0, kvc, blk, policy);
                tma_load_4d(ring_s + (2 * s + 1) * C::TILE, &vmap, full, 16 * sub, 0, kvc, blk,
                            policy);
              } else {
                // Row num_blocks * block_size is wholly out of bounds: TMA fills zeros.
                const int row0 = bad ? a.num_blocks * a.block_size : tile_row(a, phys, b + j);
                if constexpr (!KV8) {  // grouped view: 8-token groups, 128-byte swizzle
                  tma_load_5d(ring_s + (2 * s) * C::TILE, &kmap, full, 0, 0, 0, row0 / 8, kvh, policy);
                  tma_load_5d(ring_s + (2 * s + 1) * C::TILE, &vmap, full, 0, 0, 0, row0 / 8, kvh,
                              policy);
                } else {  // e4m3: swizzled 3-D view, one tile (PAIR: two kv heads) per copy
                  const int kh = C::PAIR ? 2 * kvh : kvh;
                  tma_load_3d(ring_s + (2 * s) * C::TILE, &kmap, full, 0, kh, row0, policy);
                  tma_load_3d(ring_s + (2 * s + 1) * C::TILE, &vmap, full, 0, kh, row0, policy);
                }
              }
            } else {
              mbar_arrive(full);
            }
          }
          ok = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
          ++pos;
        }
        t += seg_n;
        b += seg_n;
        ++seg;
        if (b == nb && t < hi) {  // next (request, kv head) pair
          b = 0;
          if (++kvh == a.num_kv_heads) {
            kvh = 0;
            base += static_cast<long long>(nb) * a.num_kv_heads;
            nb = 0;
            while (nb == 0 && ++r < a.num_seqs) {
              if (r == nxt_r) {
                nb = blocks_from(a, r, nxt_len, nxt_q0, nxt_q1, &len, &row);
#pragma unroll
                for (int m = 0; m < kRowCache; ++m) cur_ids[m] = nxt_ids[m];
              } else {
                nb = request_blocks(a, r, &len, &row);
                load_row(r, cur_ids);
              }
            }
            if (nb == 0) ok = false;  // cannot happen while t < hi
            else prefetch_next(r);
          }
        }
      }
    }
    // One "done" stage for each consumer warp.
    for (int j = 0; j < C::NC; ++j) {
      if (lane == 0 && stage_begin(pos)) {
        const int s = pos % C::STAGES;
        meta[s] = make_int2(0, kDone);
        mbar_arrive(full0 + 8 * s);
      }
      ++pos;
    }
    if (lane == 0 && *abort_flag) {
      // Let copies already in flight land before the CTA can exit.
      for (int i = max(0, pos - C::STAGES); i < pos; ++i)
        (void)mbar_wait(full0 + 8 * (i % C::STAGES), (i / C::STAGES) & 1);
      for (int k = 0; k < 2; ++k) (void)mbar_wait(qfull0 + 8 * k, 0);
    }
    // Deferred dependency: the CTA completes only after the previous grid.
    if (a.defer_griddep && lane == 0) griddep_wait();
    return;
  }

  if (warp == C::NC + 1) {
    // ================================================================ epilogue
    // Finishes each segment handed over by the consumers: the bf16 output of
    // a whole (request, kv head) pair, or the partial of a shared pair, its
    // pair counter and, for the last contributor, the merge of all partials.
    const float* hr = reinterpret_cast<const float*>(smem + C::OFF_HAND);
    for (int seg = 0;; ++seg) {
      const int got = mbar_wait(hfull0, seg & 1) ? 1 : 0;
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) {
          record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, 8);
          *abort_flag = 1;
        }
        break;
      }
      const SegInfo e = *reinterpret_cast<const SegInfo*>(hr + C::WF);
      if (e.kind == kEndSeg) break;
      const int head0 = e.kvh * a.group;
      if (e.kind == kWhole) {
        for (int it = lane; it < a.group * (D / 2); it += 32) {
          const int h = it / (D / 2);
          const int d = (it % (D / 2)) * 2;
          const float inv = a.v_scale / hr[GMAX * D + 2 * h + 1];
          const float2 ov = *reinterpret_cast<const float2*>(hr + h * D + d);
          *reinterpret_cast<__nv_bfloat162*>(
              a.out + (static_cast<size_t>(e.row) * a.num_heads + head0 + h) * D + d) =
              __floats2bfloat162_rn(ov.x * inv, ov.y * inv);
        }
      } else {
        const int pslot = e.kind == kTail ? 1 : 0;
        const long long W = *total_tiles;
        const int nsplit = MIX ? *split_ctas : a.num_ctas;
        const int c0 = cta_of_tile(W, nsplit, e.t0);
        const int c1 = cta_of_tile(W, nsplit, e.t0 + e.nblk - 1);
        unsigned long long* counter = a.counters + static_cast<size_t>(e.r) * a.num_kv_heads + e.kvh;
        // If every other contributor has already counted (the usual case for
        // the CTA whose range ends inside the pair, at the end of its work),
        // merge now from this CTA's own record, without publishing it.
        int last = 0;
        if (lane == 0 && c1 > c0 &&
            ld_acquire_u64(counter) == ((static_cast<unsigned long long>(a.epoch) << 32) |
                                        static_cast<unsigned>(c1 - c0)))
          last = 2;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last == 0) {
          for (int it = lane; it < a.group * (D / 2); it += 32) {
            const int h = it / (D / 2);
            const int d = (it % (D / 2)) * 2;
            const float M = hr[GMAX * D + 2 * h], L = hr[GMAX * D + 2 * h + 1];
            const float inv = a.v_scale / L;
            const float2 ov = *reinterpret_cast<const float2*>(hr + h * D + d);
            const size_t rec = (static_cast<size_t>(cta) * 2 + pslot) * a.group + h;
            *reinterpret_cast<float2*>(a.part_o + rec * D + d) = make_float2(ov.x * inv, ov.y * inv);
            if (d == 0) *reinterpret_cast<float2*>(a.part_ml + rec * 2) = make_float2(M, L);
          }
          // Publish the partial; the last of the pair's contributors merges them.
          __threadfence();
          __syncwarp();
          if (lane == 0) last = contribute(counter, a.epoch, c1 - c0 + 1, a.status, e.r) ? 1 : 0;
          last = __shfl_sync(0xffffffffu, last, 0);
        }
        if (last) {
          __syncwarp();  // lane 0 saw the other contributors' counts
          __threadfence();
          // Lane L merges head_dim pairs L, L + 32, ... of every head.  The
          // loads of one contributor are independent of each other, so each
          // contributor costs one memory round trip.
          constexpr int kPer = GMAX * D / 2 / 32;  // head_dim pairs per lane (all heads)
          float M[GMAX], L[GMAX], o[kPer][2];
#pragma unroll
          for (int h = 0; h < GMAX; ++h) {
            M[h] = kNegBig;
            L[h] = 0.f;
          }
#pragma unroll
          for (int k = 0; k < kPer; ++k) o[k][0] = o[k][1] = 0.f;
          for (int c = c0; c <= c1; ++c) {
            const size_t rec0 = (static_cast<size_t>(c) * 2 + (c == c0 ? 1 : 0)) * a.group;
            float2 ml[GMAX], ov[kPer];
#pragma unroll
            for (int h = 0; h < GMAX; ++h) ml[h] = make_float2(kNegBig, 0.f);
#pragma unroll
            for (int k = 0; k < kPer; ++k) ov[k] = make_float2(0.f, 0.f);
            const bool own = last == 2 && c == cta;  // this CTA's record is still in shared memory
#pragma unroll
            for (int h = 0; h < GMAX; ++h)
              if (h < a.group)
                ml[h] = own ? make_float2(hr[GMAX * D + 2 * h], hr[GMAX * D + 2 * h + 1])
                            : __ldcg(reinterpret_cast<const float2*>(a.part_ml + (rec0 + h) * 2));
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
              const int h = (lane + 32 * k) / (D / 2), d = ((lane + 32 * k) % (D / 2)) * 2;
              if (h >= a.group) continue;
              if (own) {
                const float2 u = *reinterpret_cast<const float2*>(hr + h * D + d);
                const float inv = a.v_scale / ml[h].y;
                ov[k] = make_float2(u.x * inv, u.y * inv);
              } else {
                ov[k] = __ldcg(reinterpret_cast<const float2*>(a.part_o + (rec0 + h) * D + d));
              }
            }
            float wo[GMAX], wt[GMAX];
#pragma unroll
            for (int h = 0; h < GMAX; ++h) {
              if (h >= a.group) continue;
              const float mx = fmaxf(M[h], ml[h].x);
              wo[h] = fast_exp2(M[h] - mx);
              wt[h] = ml[h].y * fast_exp2(ml[h].x - mx);
              L[h] = L[h] * wo[h] + wt[h];
              M[h] = mx;
            }
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
              const int h = (lane + 32 * k) / (D / 2);
              if (h >= a.group) continue;
              o[k][0] = o[k][0] * wo[h] + wt[h] * ov[k].x;
              o[k][1] = o[k][1] * wo[h] + wt[h] * ov[k].y;
            }
          }
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const int h = (lane + 32 * k) / (D / 2), d = ((lane + 32 * k) % (D / 2)) * 2;
            if (h >= a.group) continue;
            const float inv = 1.f / L[h];
            *reinterpret_cast<__nv_bfloat162*>(
                a.out + (static_cast<size_t>(e.row) * a.num_heads + head0 + h) * D + d) =
                __floats2bfloat162_rn(o[k][0] * inv, o[k][1] * inv);
          }
          if (lane == 0) release_pair(counter);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(hempty0);
    }
    return;
  }

  // ================================================================ consumers
  // lane = 4 fg + ft in the m16n8k16 fragments; the 8 columns of every
  // product are q heads (those >= group are zero).
  const int fg = lane >> 2, ft = lane & 3;
  uint32_t qf[C::KS][2];  // q^T fragments: head fg, head_dim 16 ks + 2 ft (+1, +8, +9)
  float om[C::KS][4];     // O^T: head_dim 16 m + fg (+8) (e4m3: 16 m + 2 fg (+1)) x heads 2 ft (+1)
  float mh[2] = {kNegBig, kNegBig};  // running max (log2 units) of heads 2 ft, 2 ft + 1
  float lh[2] = {0.f, 0.f};          // this lane's share of their exp-sums
  SegInfo si{};
  bool fresh = true;
  int seg = 0;
  // Barrier of the consumer warps: lane 0 of each warp arrives, every
  // lane waits (bounded); orders the warps' shared-memory writes before the
  // reads after it.  Returns false (and flags an abort) on a timeout.
  uint32_t cphase = 0;
  auto csync = [&]() -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(csync_bar);
    const int ok = mbar_wait(csync_bar, cphase & 1) ? 1 : 0;
    ++cphase;
    if (__all_sync(0xffffffffu, ok)) return true;
    if (lane == 0) {
      record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, 7);
      *abort_flag = 1;
    }
    return false;
  };

  // No abort check per stage: every wait below is bounded on its own.
  for (int pos = warp;; pos += C::NC) {
    const int s = pos % C::STAGES;
    const int landed = mbar_wait(full0 + 8 * s, (pos / C::STAGES) & 1) ? 1 : 0;
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) {
        record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, 2);
        *abort_flag = 1;
      }
      break;
    }
    const int2 m = meta[s];
    if (m.y & kDone) {
      if (warp == 0) {  // tell the epilogue warp that no segment follows
        const int ok = (seg < 1 || mbar_wait(hempty0, (seg - 1) & 1)) ? 1 : 0;
        if (__all_sync(0xffffffffu, ok)) {
          if (lane == 0) {
            SegInfo* rec = reinterpret_cast<SegInfo*>(reinterpret_cast<float*>(smem + C::OFF_HAND) +
                                                      C::WF);
            rec->kind = kEndSeg;
            mbar_arrive(hfull0);
          }
        } else if (lane == 0) {
          record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, 10);
          *abort_flag = 1;
        }
      }
      break;
    }

    if (fresh) {  // first stage of a segment: take its q and reset the state
      const int slot = seg & 1;
      const int qok = mbar_wait(qfull0 + 8 * slot, (seg >> 1) & 1) ? 1 : 0;
      if (!__all_sync(0xffffffffu, qok)) {
        if (lane == 0) {
          record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, 5);
          *abort_flag = 1;
        }
        break;
      }
      si = seginfo[slot];
      const uint32_t qs = qbuf_s + slot * (GMAX * D * 2);
      // q stays bf16 (f16 for e4m3 caches; the products are exact in fp32);
      // the scale is applied to the fp32 scores.
#pragma unroll
      for (int ks = 0; ks < C::KS; ++ks)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if constexpr (KV8) {
            // head_dim in the order the e4m3 K fragments hold it: product
            // index 2 ft (+1) is element 4 ft (+1) of the 16-wide step,
            // 2 ft + 8 (+9) is element 4 ft + 2 (+3).
            const uint32_t w =
                fg < a.group ? ld_shared_u32(qs + (fg * D + 16 * ks + 4 * ft + 2 * j) * 2) : 0u;
            qf[ks][j] = pack_f16x2_sat(bf16_lo(w), bf16_hi(w));
          } else {
            qf[ks][j] =
                fg < a.group ? ld_shared_u32(qs + (fg * D + 16 * ks + 8 * j + 2 * ft) * 2) : 0u;
          }
        }
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty0 + 8 * slot);
#pragma unroll
      for (int mt = 0; mt < C::KS; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) om[mt][i] = 0.f;
      mh[0] = mh[1] = kNegBig;
      lh[0] = lh[1] = 0.f;
      fresh = false;
    }

    if (!(m.y & kSkip)) {
      const uint32_t kt = ring_s + (2 * s) * C::TILE;
      const uint32_t vt = kt + C::TILE;
      const int tok0 = m.x * kBlockSize;
      const int seq_len = si.seq_len;
      // S^T (16 tokens x 8 heads) = K q^T.  Matrix mi = lane / 8 of each
      // ldmatrix: tokens 8 (mi % 2) .. + 7, head_dim chunk 2 ks + mi / 2.
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      const int ka_t = ((lane >> 3) & 1) * 8 + (lane & 7);
      if constexpr (C::PAIR) {
        // Two kv heads: S^T of each against all 8 q heads; a lane keeps the
        // one its heads 2 ft, 2 ft + 1 belong to (kv head ft / 2).
        float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int kp = 0; kp < C::KS / 2; ++kp) {
            uint32_t r8[4];
            ldsm_x4(kt + e8_row_offset(2 * ka_t + hh, 2 * kp + (lane >> 4)), r8);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t af[4] = {e4m3x2_f16x2(r8[2 * h]), e4m3x2_f16x2(r8[2 * h + 1]),
                                      e4m3x2_f16x2(r8[2 * h] >> 16), e4m3x2_f16x2(r8[2 * h + 1] >> 16)};
              mma_16816_f16(s2[hh], af, qf[2 * kp + h][0], qf[2 * kp + h][1]);
            }
          }
#pragma unroll
        for (int i = 0; i < 4; ++i) sacc[i] = ft < 2 ? s2[0][i] : s2[1][i];
      } else if constexpr (KV8) {
        // One ldmatrix covers two 16-wide steps of e4m3 head_dim: matrix mi
        // = tokens 8 (mi % 2) .., chunk 2 kp + mi / 2; a lane's register
        // holds elements 4 ft .. 4 ft + 3 of its token's chunk.
#pragma unroll
        for (int kp = 0; kp < C::KS / 2; ++kp) {
          uint32_t r8[4];
          const int c8 = 2 * kp + (lane >> 4);
          ldsm_x4(kt + (XS ? static_cast<uint32_t>(c8 * 256 + xs8_token(ka_t) * 16)
                           : e8_offset<D>(ka_t, c8)),
                  r8);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t af[4] = {e4m3x2_f16x2(r8[2 * h]), e4m3x2_f16x2(r8[2 * h + 1]),
                                    e4m3x2_f16x2(r8[2 * h] >> 16), e4m3x2_f16x2(r8[2 * h + 1] >> 16)};
            mma_16816_f16(sacc, af, qf[2 * kp + h][0], qf[2 * kp + h][1]);
          }
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < C::KS; ++ks) {
          uint32_t af[4];
          const int c = 2 * ks + (lane >> 4);
          ldsm_x4(kt + (XS ? xs_k_offset(ka_t, c) : grp_offset<D>(ka_t, c)), af);
          mma_16816(sacc, af, qf[ks][0], qf[ks][1]);
        }
      }
      // Scores in log2 units: (token fg (+8), head 2 ft (+1)); tokens past
      // seq_len and padding heads get weight 0.
      float p[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int srow = fg + (i >> 1) * 8;
        const int stok = (KV8 && XS) ? xs8_token(srow) : srow;
        const bool ok = tok0 + stok < seq_len && 2 * ft + (i & 1) < a.group;
        p[i] = ok ? sacc[i] * a.scale_log2 : -INFINITY;
      }
      // The tile maximum of each head over the 8 lanes that share ft.  bf16
      // token-major: a warp reduction of order-preserving keys per group of
      // lanes (faster than a chain of shuffles there: 115.3 -> 113.4 us on
      // the 8B batch); e4m3 and x-split: shuffles (the reduction measured
      // 90.9 -> 104.9 us on e4m3, 437 -> 491 us on the x-split 70B batch).
      float tmax[2] = {fmaxf(p[0], p[2]), fmaxf(p[1], p[3])};
      if constexpr (KV8 || XS) {
#pragma unroll
        for (int bb = 4; bb < 32; bb <<= 1) {
          tmax[0] = fmaxf(tmax[0], __shfl_xor_sync(0xffffffffu, tmax[0], bb));
          tmax[1] = fmaxf(tmax[1], __shfl_xor_sync(0xffffffffu, tmax[1], bb));
        }
      } else {
        const unsigned ftmask = 0x11111111u << ft;
#pragma unroll
        for (int i = 0; i < 2; ++i)
          tmax[i] = max_key_to_float(__reduce_max_sync(ftmask, float_to_max_key(tmax[i])));
      }
      if (__any_sync(0xffffffffu,
                     tmax[0] > mh[0] + kRescaleSlack || tmax[1] > mh[1] + kRescaleSlack)) {
        float al[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float mn = fmaxf(mh[e], tmax[e]);
          al[e] = fast_exp2(mh[e] - mn);
          mh[e] = mn;
          lh[e] *= al[e];
        }
#pragma unroll
        for (int mt = 0; mt < C::KS; ++mt) {
          om[mt][0] *= al[0];
          om[mt][1] *= al[1];
          om[mt][2] *= al[0];
          om[mt][3] *= al[1];
        }
      }
      // Weights rounded to bf16 (f16 for e4m3 caches) for the product; l
      // sums the rounded values.
#pragma unroll
      for (int i = 0; i < 4; ++i) p[i] = fast_exp2(p[i] - mh[i & 1]);
      uint32_t pk0, pk1;
      if constexpr (KV8) {
        pk0 = pack_f16x2_sat(p[0], p[1]);  // token fg:     heads 2 ft, 2 ft + 1
        pk1 = pack_f16x2_sat(p[2], p[3]);  // token fg + 8
        lh[0] += f16_lo(pk0) + f16_lo(pk1);
        lh[1] += f16_hi(pk0) + f16_hi(pk1);
      } else {
        pk0 = pack_bf16x2(p[0], p[1]);
        pk1 = pack_bf16x2(p[2], p[3]);
        lh[0] += bf16_lo(pk0) + bf16_lo(pk1);
        lh[1] += bf16_hi(pk0) + bf16_hi(pk1);
      }
      const uint32_t pb0 = movmatrix_t(pk0);  // P^T: tokens 2 ft, 2 ft + 1 of head fg
      const uint32_t pb1 = movmatrix_t(pk1);  // tokens 2 ft + 8, 2 ft + 9
      // O^T (head_dim x 8 heads) += V^T P^T, 16 head_dim rows per product.
      // In the last block of a request the V rows past seq_len may hold NaN
      // (0 x NaN is NaN): their halves of the V^T fragments are cleared.
      uint32_t vm01 = 0xffffffffu, vm89 = 0xffffffffu;
      if (tok0 + kBlockSize > seq_len) {
        // The two token pairs a lane's V^T halves hold: (2 ft, 2 ft + 1) and
        // (2 ft + 8, 2 ft + 9); e4m3 x-split: (4 ft, 4 ft + 1), (4 ft + 2, 4 ft + 3).
        const int t0 = tok0 + ((KV8 && XS) ? 4 * ft : 2 * ft);
        const int t8 = t0 + ((KV8 && XS) ? 2 : 8);
        vm01 = (t0 < seq_len ? 0x0000ffffu : 0u) | (t0 + 1 < seq_len ? 0xffff0000u : 0u);
        vm89 = (t8 < seq_len ? 0x0000ffffu : 0u) | (t8 + 1 < seq_len ? 0xffff0000u : 0u);
      }
      const int va_r = lane & 7, va_m = lane >> 3;
      if constexpr (KV8 && XS) {
        // e4m3 x-split V^T: plain ldmatrix of 8 head_dim rows of 16 bytes;
        // matrix mi = head_dim 16 (2 mp + mi / 2) + 8 (mi % 2) ..  A lane's
        // register holds tokens 4 ft .. 4 ft + 3 of row fg: its low half is
        // reduction index (2 ft, 2 ft + 1), its high half (2 ft + 8, 2 ft + 9).
#pragma unroll
        for (int mp = 0; mp < C::KS / 2; ++mp) {
          uint32_t r8[4];
          ldsm_x4(vt + static_cast<uint32_t>((16 * (2 * mp + (va_m >> 1)) + 8 * (va_m & 1) + va_r) * 16),
                  r8);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t af[4] = {e4m3x2_f16x2(r8[2 * h]) & vm01, e4m3x2_f16x2(r8[2 * h + 1]) & vm01,
                                    e4m3x2_f16x2(r8[2 * h] >> 16) & vm89,
                                    e4m3x2_f16x2(r8[2 * h + 1] >> 16) & vm89};
            mma_16816_f16(om[2 * mp + h], af, pb0, pb1);
          }
        }
      } else if constexpr (C::PAIR) {
        // Two kv heads: O^T += V_h^T P_h^T for each, P_h^T the weights of
        // kv head h's q heads (B operand column fg = q head: fg / 4 = h).
        const uint32_t pq0[2] = {fg < 4 ? pb0 : 0u, fg < 4 ? 0u : pb0};
        const uint32_t pq1[2] = {fg < 4 ? pb1 : 0u, fg < 4 ? 0u : pb1};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int mp = 0; mp < C::KS / 2; ++mp) {
            uint32_t r8[4];
            ldsm_x4_t(vt + e8_row_offset(2 * (8 * (va_m & 1) + va_r) + hh, 2 * mp + (va_m >> 1)), r8);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t lo = bytes_0213(r8[2 * h]), hi = bytes_0213(r8[2 * h + 1]);
              uint32_t af[4] = {e4m3x2_f16x2(lo), e4m3x2_f16x2(lo >> 16), e4m3x2_f16x2(hi),
                                e4m3x2_f16x2(hi >> 16)};
              af[0] &= vm01;
              af[1] &= vm01;
              af[2] &= vm89;
              af[3] &= vm89;
              mma_16816_f16(om[2 * mp + h], af, pq0[hh], pq1[hh]);
            }
          }
      } else if constexpr (KV8) {
        // e4m3 V^T: matrix mi = tokens 8 (mi % 2) .., chunk 2 mp + mi / 2,
        // read transposed in 16-bit units; a lane's register holds (token
        // 2 ft, 2 ft + 1) x (head_dim 2 fg, 2 fg + 1) of the chunk.  Byte
        // permute + conversion give row fg (head_dim 2 fg) and row fg + 8
        // (head_dim 2 fg + 1) of the 16-row product, tokens 2 ft, 2 ft + 1.
#pragma unroll
        for (int mp = 0; mp < C::KS / 2; ++mp) {
          uint32_t r8[4];
          ldsm_x4_t(vt + e8_offset<D>(8 * (va_m & 1) + va_r, 2 * mp + (va_m >> 1)), r8);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t lo = bytes_0213(r8[2 * h]), hi = bytes_0213(r8[2 * h + 1]);
            uint32_t af[4] = {e4m3x2_f16x2(lo), e4m3x2_f16x2(lo >> 16), e4m3x2_f16x2(hi),
                              e4m3x2_f16x2(hi >> 16)};
            af[0] &= vm01;
            af[1] &= vm01;
            af[2] &= vm89;
            af[3] &= vm89;
            mma_16816_f16(om[2 * mp + h], af, pb0, pb1);
          }
        }
      } else {
#pragma unroll
      for (int mt = 0; mt < C::KS; ++mt) {
        uint32_t af[4];
        if constexpr (XS) {
          // V^T rows: matrix mi = head_dim 16 mt + 8 (mi % 2) .., tokens 8 (mi / 2) ..
          ldsm_x4(vt + xs_v_offset(16 * mt + 8 * (va_m & 1) + va_r, va_m >> 1), af);
        } else {
          // token rows, transposed: matrix mi = tokens 8 (mi / 2) .., chunk 2 mt + mi % 2
          ldsm_x4_t(vt + grp_offset<D>(8 * (va_m >> 1) + va_r, 2 * mt + (va_m & 1)), af);
        }
        af[0] &= vm01;
        af[1] &= vm01;
        af[2] &= vm89;
        af[3] &= vm89;
        mma_16816(om[mt], af, pb0, pb1);
      }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
    if (!(m.y & kLastRow)) continue;

    // ======================== end of segment: merge the two warps' states
    // and hand the result to the epilogue warp.  Record: O^T accumulators
    // [GMAX][D], (m, l) per head, the segment record; each lane writes and
    // reads only its own (head, d) places.
    float ls[2] = {lh[0], lh[1]};
#pragma unroll
    for (int bb = 4; bb < 32; bb <<= 1) {
      ls[0] += __shfl_xor_sync(0xffffffffu, ls[0], bb);
      ls[1] += __shfl_xor_sync(0xffffffffu, ls[1], bb);
    }
    float* hrec = reinterpret_cast<float*>(smem + C::OFF_HAND);
    // head_dim row of accumulator om[mt][i] (the e4m3 V^T fragments
    // interleave the rows: product row fg is 2 fg, row fg + 8 is 2 fg + 1).
    auto orow = [&](int mt, int i) -> int {
      return (KV8 && !XS) ? 16 * mt + 2 * fg + (i >> 1) : 16 * mt + fg + 8 * (i >> 1);
    };
    auto put = [&]() {
#pragma unroll
      for (int mt = 0; mt < C::KS; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = 2 * ft + (i & 1);
          if (h < a.group) hrec[h * D + orow(mt, i)] = om[mt][i];
        }
      if (fg == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int h = 2 * ft + e;
          if (h < a.group) {
            hrec[GMAX * D + 2 * h] = mh[e];
            hrec[GMAX * D + 2 * h + 1] = ls[e];
          }
        }
      }
    };
    if (warp == 1) {
      // The record was last handed over one segment ago.
      const int ok = (seg < 1 || mbar_wait(hempty0, (seg - 1) & 1)) ? 1 : 0;
      if (__all_sync(0xffffffffu, ok)) {
        put();
      } else if (lane == 0) {
        record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, 9);
        *abort_flag = 1;
      }
    }
    if (!csync() || *abort_flag) break;
    if (warp == 0) {
      // Merge warp 1's state into this warp's, then hand the segment over.
      float wa[2], wb[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * ft + e;
        const float mo = h < a.group ? hrec[GMAX * D + 2 * h] : kNegBig;
        const float lo = h < a.group ? hrec[GMAX * D + 2 * h + 1] : 0.f;
        const float mx = fmaxf(mh[e], mo);
        wa[e] = fast_exp2(mh[e] - mx);
        wb[e] = fast_exp2(mo - mx);
        mh[e] = mx;
        ls[e] = ls[e] * wa[e] + lo * wb[e];
      }
#pragma unroll
      for (int mt = 0; mt < C::KS; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = 2 * ft + (i & 1);
          const float ov = h < a.group ? hrec[h * D + orow(mt, i)] : 0.f;
          om[mt][i] = om[mt][i] * wa[i & 1] + ov * wb[i & 1];
        }
      __syncwarp();  // every lane has read the (m, l) entries before they change
      put();
      if (lane == 0) *reinterpret_cast<SegInfo*>(hrec + C::WF) = si;
      __syncwarp();
      if (lane == 0) mbar_arrive(hfull0);
    }
    fresh = true;
    ++seg;
  }
}

template <int D, int GMAX, bool KV8, bool XS, bool MIX = false>
cudaError_t launch_decode_impl(const DecodeArgs& a, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, cudaStream_t stream) {
  using C = DecodeCfg<D, GMAX, KV8, XS>;
  auto* kernel = paged_decode_kernel<D, GMAX, KV8, XS, MIX>;
  static bool attr_set[64] = {false};  // per device: set once
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  return launch_overlapped(kernel, dim3(a.num_ctas), dim3(C::THREADS), C::SMEM, stream, kmap,
                           vmap, a);
}

}  // namespace

int decode_gmax(int group) {
  if (group <= 1) return 1;
  if (group <= 2) return 2;
  if (group <= 4) return 4;
  return 0;
}

int decode_ctas_per_sm(int head_dim, int group) {
  const int gmax = decode_gmax(group);
#define PA_DECODE_CASE(DD, GG) \
  if (head_dim == DD && gmax == GG) return DecodeCfg<DD, GG>::MINB;
  PA_DECODE_CASE(128, 1) PA_DECODE_CASE(128, 2) PA_DECODE_CASE(128, 4)
  PA_DECODE_CASE(64, 1) PA_DECODE_CASE(64, 2) PA_DECODE_CASE(64, 4)
#undef PA_DECODE_CASE
  return 1;
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          int head_dim, bool kv8, bool xsplit, cudaStream_t stream) {
  // e4m3 units of two kv heads (8 q heads, head_dim 128): one instantiation.
  if (kv8 && !xsplit && a.group == 8 && head_dim == 128 && a.tile_sms == 0)
    return launch_decode_impl<128, 8, true, false>(a, kmap, vmap, stream);
  const int gmax = decode_gmax(a.group);
  const bool mix = a.tile_sms > 0;  // built for head_dim 128 (the host splits the SMs only there)
#define PA_DECODE_CASE(DD, GG)                                                      \
  if (head_dim == DD && gmax == GG)                                                 \
    return kv8 ? (xsplit ? launch_decode_impl<DD, GG, true, true>(a, kmap, vmap, stream)      \
                  : mix    ? launch_decode_impl<DD, GG, true, false, DD == 128>(a, kmap, vmap, stream) \
                           : launch_decode_impl<DD, GG, true, false>(a, kmap, vmap, stream))    \
               : (xsplit ? launch_decode_impl<DD, GG, false, true>(a, kmap, vmap, stream)     \
                  : mix    ? launch_decode_impl<DD, GG, false, false, DD == 128>(a, kmap, vmap, stream) \
                           : launch_decode_impl<DD, GG, false, false>(a, kmap, vmap, stream));
  PA_DECODE_CASE(128, 1) PA_DECODE_CASE(128, 2) PA_DECODE_CASE(128, 4)
  PA_DECODE_CASE(64, 1) PA_DECODE_CASE(64, 2) PA_DECODE_CASE(64, 4)
#undef PA_DECODE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
