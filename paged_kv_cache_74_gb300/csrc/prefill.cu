// prefill.cu -- chunked-prefill attention of a varlen batch on the sm_103a
// tensor cores (tcgen05).
//
// Method ("分块预填充与混合批处理", section 11.6; "vLLM 深度解析（二）：
// PagedAttention 核心机制", sections 2.1, 2.2, 3.1, 3.2.9 and 5.2): request r
// owns query rows query_start_loc[r] .. query_start_loc[r+1] - 1; with q_len
// rows and K/V length seq_len, row i sits at position ctx + i (ctx = seq_len
// - q_len) and attends keys 0 .. ctx + i, read through the block table.
// O = softmax(scale * Q K^T) V is computed 128 keys at a time with the
// online softmax state (m, l) per row; S and P never reach HBM.  Pieces of a
// row's keys computed by different CTAs are merged through their (m_j, l_j,
// O_j): m = max m_j, L = sum l_j 2^(m_j - m), O = sum O_j l_j 2^(m_j - m) / L.
//
// GB300 design.
// * Work unit: 128 query rows of one request for TWO q heads of the same kv
//   head (slots 0 and 1; one head when the group has an odd head left).
//   Every K/V tile is copied into shared memory once and serves both heads.
// * Persistent grid, one CTA per SM.  The 128-key steps of all units are
//   numbered (request-major; within a request the last query tile, which
//   sees the most keys, first; then head pair; then key step) and cut into
//   equal contiguous ranges, one per CTA, so every SM gets the same number
//   of MMA steps whatever the mix of chunk lengths.  A unit cut by a range
//   boundary is finished by whichever of its contributors counts last on
//   an epoch-tagged counter: it merges the pieces' partials.
// * A small tile batch with decode rows behind it (`partition`) is cut over
//   fewer CTAs, tile_kernel_sms() of them, the tile work's share of the
//   batch's estimated SM time; the other CTAs exit at once and leave their
//   SMs to the decode CTAs of the same call, which then stream next to the
//   tiles instead of after them.
// * Per step and slot b: S_b = Q_b K^T (M = N = 128, K = head_dim) into TMEM
//   columns [128 b, 128 b + 128); the softmax warps of slot b read S_b, write
//   P_b = 2^(S_b * scale * log2 e - m) as bf16 over the first 64 of those
//   columns, and O_b += P_b V (A = P_b read from TMEM, B = V from shared
//   memory, MN-major) accumulates in TMEM columns 256 + b * head_dim.  The
//   MMA warp issues P_0 V, then S_0 of the next step, then P_1 V, then S_1
//   of the next step: while the tensor core works for one slot the other
//   slot's softmax runs (ping-pong).
// * The reference m of a row moves only when a step's maximum exceeds it by
//   more than 2^8; O (in TMEM) and l are rescaled then (S_b completing
//   implies the P_b V before it has completed, so O_b is current).
// * Warp roles (352 threads): warp 0 Q and K producer (TMA; each 16-token
//   block of a 128-key tile is one copy that lands as [8-key group][head_dim
//   half][8 keys][128 B], the layout both MMAs read) and the range walk;
//   warp 10 V producer; warp 1 MMA issuer; warps 2-5 softmax of slot 0 and
//   warps 6-9 of slot 1 (thread = query row, all 128 columns of S), which
//   also write the output, the partials and the merge.
// V rows of keys that are out of context or were not loaded are zeroed
// before the P.V product (a zero weight does not cancel a NaN inside the
// MMA).  Every wait is bounded; a timeout records PA_DEV_WAIT_TIMEOUT.
#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "work_split.cuh"

namespace pa {
namespace {

constexpr float kNegBigP = -1e30f;
constexpr float kRescaleSlackP = 8.0f;  // log2 units
constexpr int kSegWhole = 0;            // the whole unit: bf16 output
constexpr int kSegHead = 1;             // continues a unit begun by an earlier CTA: partial slot 0
constexpr int kSegTail = 2;             // begins a unit finished by later CTAs: partial slot 1
constexpr int kSegEnd = 3;              // no more work
// How long a unit's first CTA waits for the unit's other pieces before it
// publishes its own instead of merging them.
constexpr unsigned long long kMergeWaitNs = 20000;

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Two floats rounded to bf16 (nearest even), packed low / high.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

template <int D>
struct PrefillCfg {
  static constexpr int BM = 128;                    // query rows per unit
  static constexpr int BN = 128;                    // keys per step (8 blocks of 16)
  static constexpr int HALVES = D / 64;             // 128-byte column chunks of head_dim
  static constexpr int CHUNK = 128 * 128;           // 128 rows x 128 bytes, swizzled
  static constexpr int QBYTES = HALVES * CHUNK;     // Q of one head
  static constexpr int TBYTES = HALVES * CHUNK;     // K (or V) of one step
  static constexpr int BLOCK_BYTES = HALVES * 16 * 128;  // K (or V) of one 16-token block
  // K and V blocks land as [8-key group][head_dim half][8 keys][128 B]: the
  // 8-key groups of a tile are GSTRIDE apart, head_dim halves 1 KB apart.
  static constexpr int GSTRIDE = HALVES * 1024;
  static constexpr int NST = D == 128 ? 2 : 4;      // K stages = V stages
  static constexpr int SEGS = 4;                    // segment records in flight
  static constexpr int SEG_INTS = 16;
  static constexpr int OFF_Q = 0;                   // [2 slots]
  static constexpr int OFF_K = OFF_Q + 2 * QBYTES;
  static constexpr int OFF_V = OFF_K + NST * TBYTES;
  static constexpr int OFF_SEG = OFF_V + NST * TBYTES;
  static constexpr int REQ_CACHE = 256;             // requests whose lengths are cached
  static constexpr int OFF_REQ = OFF_SEG + SEGS * SEG_INTS * 4;  // [3][REQ_CACHE] ints
  static constexpr int OFF_BAR = OFF_REQ + 3 * REQ_CACHE * 4;
  static constexpr int NBAR = 4 * NST + 12 + 2 * SEGS + 2 + 22 + 2 * NST + 2;
  // e4m3 cache: a step's K (or V) bytes land as 16-token blocks of head_dim
  // bytes in the upper half of the f16 stage they are converted into.
  static constexpr int RAW_BLOCK = 16 * D;
  static constexpr int RAW_OFF = TBYTES / 2;
  // Merge staging at a CTA's last segment: slot b's Q buffer and one K/V
  // ring (K for slot 0, V for slot 1) are free once O_b is final; they are
  // cut into 16 KB buffers (32 columns of one partial record), the last one
  // holding the (m, l) records of up to MREM contributors.
  static constexpr int MBUF = 16384;
  static constexpr int MQB = QBYTES / MBUF;                       // buffers in the Q buffer
  static constexpr int MDATA = (QBYTES + NST * TBYTES) / MBUF - 1;  // partial O buffers
  static constexpr int MREM = MBUF / (128 * 8);                   // (m, l) records that fit
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;  // + 1024-byte alignment slack
  static constexpr int THREADS = 11 * 32;
  static constexpr uint32_t TMEM_COLS = 512;         // S0 0, S1 128, O0 256, O1 256 + D
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0);
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 1);
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(MDATA >= 2 && MDATA <= 5 && D % 32 == 0, "merge staging");
};

// Barrier indices.
template <int NST, int SEGS>
struct PBars {
  static constexpr int KFULL = 0;                // [NST] K step landed
  static constexpr int KFREE = KFULL + NST;      // [NST] both S MMAs that read it are done
  static constexpr int VFULL = KFREE + NST;      // [NST]
  static constexpr int VFREE = VFULL + NST;      // [NST] both P.V MMAs that read it are done
  static constexpr int QFULL = VFREE + NST;      // [2] Q of a slot landed
  static constexpr int QFREE = QFULL + 2;        // [2] last S MMA of a segment read it
  static constexpr int SFULL = QFREE + 2;        // [2] S_b in TMEM
  static constexpr int PFULL = SFULL + 2;        // [2] P_b in TMEM (4 softmax warps)
  static constexpr int OFULL = PFULL + 2;        // [2] last P.V of a segment done
  static constexpr int OFREE = OFULL + 2;        // [2] O_b read at a segment end (4 warps)
  static constexpr int SEGFULL = OFREE + 2;      // [SEGS] segment record written
  static constexpr int SEGFREE = SEGFULL + SEGS; // [SEGS] every role is done with it
  static constexpr int SYNC = SEGFREE + SEGS;    // the 8 softmax warps
  static constexpr int DRAIN = SYNC + 1;         // the MMA warp's last commit
  static constexpr int MFULL = DRAIN + 1;        // [2][5] staged partial O chunk landed
  static constexpr int MLFULL = MFULL + 10;      // [2] staged (m, l) records landed
  static constexpr int MEMPTY = MLFULL + 2;      // [2][5] the slot's 4 warps have read a staged chunk
  static constexpr int KRAW = MEMPTY + 10;       // [NST] e4m3 K step landed (then converted)
  static constexpr int VRAW = KRAW + NST;        // [NST] e4m3 V step landed
  static constexpr int QCONV = VRAW + NST;       // [2] Q of a slot converted to f16 (4 warps)
  static constexpr int COUNT = QCONV + 2;
};

// A segment: steps [j0, j1) of one unit inside this CTA's range.
struct PSeg {
  int r, q0, row0, rows;
  int ctx, kv_end, n_kv, j0;
  int j1, h0, h1, kvh;
  int kind, unit, c0, c1;
};
static_assert(sizeof(PSeg) == 64, "segment record");

using PReq = TileReq;

__device__ __forceinline__ RowLimits row_limits(const PrefillArgs& a) {
  return RowLimits{a.max_query_len, a.max_seq_len, a.max_blocks_per_seq * a.block_size, a.total_q};
}

// From request r's query_start_loc[r], [r + 1] and seq_lens[r].
__device__ __forceinline__ PReq make_req(const PrefillArgs& a, int q0, int q1, int seq_len) {
  return tile_req(q0, q1, seq_len, row_limits(a));
}

__device__ __forceinline__ PReq prefill_req(const PrefillArgs& a, int r) {
  if (r >= a.num_seqs) return PReq{0, 0, 0, 0, 0};
  return make_req(a, __ldg(a.query_start_loc + r), __ldg(a.query_start_loc + r + 1), __ldg(a.seq_lens + r));
}

// Key steps of query tile u (u = 0: the request's last tile) of a request.
__device__ __forceinline__ int unit_steps(const PReq& p, int u, int* row0, int* rows, int* kv_end) {
  const int qt = p.ntq - 1 - u;
  *row0 = qt * 128;
  *rows = min(128, p.q_len - *row0);
  *kv_end = p.ctx + *row0 + *rows;
  return (*kv_end + 127) / 128;
}

// Key steps of all query tiles of a request (one head pair): the sum of
// unit_steps() over its tiles in closed form.
__device__ __forceinline__ int req_steps(const PReq& p) { return tile_req_steps(p); }

// Reports the prefill rows prefill_req() rejects (done once, by CTA 0).
__device__ void report_bad_prefill_rows(const PrefillArgs& a, int lane) {
  for (int r = lane; r < a.num_seqs; r += 32) {
    const int q0 = a.query_start_loc[r];
    const int q_len = a.query_start_loc[r + 1] - q0;
    if (q_len <= 1) continue;
    const int seq_len = a.seq_lens[r];
    if (q_len > seq_len || q_len > a.max_query_len || q0 < 0 || q0 + q_len > a.total_q)
      record_error(a.status, PA_DEV_BAD_QUERY_LEN, r, q_len > seq_len ? q_len : seq_len);
    else if (seq_len > a.max_seq_len || seq_len > a.max_blocks_per_seq * a.block_size)
      record_error(a.status, PA_DEV_BAD_SEQ_LEN, r, seq_len);
  }
}

// An e4m3 step (nb landed 16-token blocks of head_dim bytes at RAW_OFF of
// the stage) turned in place into the f16 operand layout the bf16 copies
// produce ([8-key group][head_dim half][8 keys][128 B], 128-byte swizzle).
// e4m3 values are exact in f16.  Run by one warp.  The 8-key groups go in
// order: group g's output bytes [g GSTRIDE, (g + 1) GSTRIDE) only cover raw
// rows of groups up to g itself (raw row t sits at RAW_OFF + t D, with
// GSTRIDE = 16 D and RAW_OFF = 128 D: the rows below (g + 1) GSTRIDE are
// t < 16 g - 112 <= 8 g + 8 for g < 16), and each group is read whole
// before it is written.
template <int D>
__device__ __forceinline__ void convert_e4m3_step(uint32_t stage, int nb, int lane) {
  using C = PrefillCfg<D>;
  constexpr int CPR = D / 16;     // 16-byte raw chunks per key row
  constexpr int KPI = 32 / CPR;   // key rows per warp-wide load
  constexpr int NLD = 8 / KPI;    // loads per lane per 8-key group
  static_assert(C::GSTRIDE == 16 * D && C::RAW_OFF == 128 * D, "in-place conversion order");
  const int c = lane % CPR;       // raw chunk: dims 16c .. 16c + 15
  const uint32_t half = (c / 4) * 1024;
  const int cc = 2 * (c % 4);     // its two f16 chunks in the half
#pragma unroll 1
  for (int g8 = 0; g8 < 2 * nb; ++g8) {
    uint4 w[NLD];
#pragma unroll
    for (int k = 0; k < NLD; ++k)
      w[k] = ld_shared_v4(stage + C::RAW_OFF + (g8 * 8 + lane / CPR + KPI * k) * D + c * 16);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < NLD; ++k) {
      const int r = lane / CPR + KPI * k;
      const uint32_t row = stage + g8 * C::GSTRIDE + half + r * 128;
      st_shared_v4(row + ((cc ^ r) * 16),
                   make_uint4(e4m3x2_to_f16x2(w[k].x), e4m3x2_to_f16x2(w[k].x >> 16),
                              e4m3x2_to_f16x2(w[k].y), e4m3x2_to_f16x2(w[k].y >> 16)));
      st_shared_v4(row + (((cc + 1) ^ r) * 16),
                   make_uint4(e4m3x2_to_f16x2(w[k].z), e4m3x2_to_f16x2(w[k].z >> 16),
                              e4m3x2_to_f16x2(w[k].w), e4m3x2_to_f16x2(w[k].w >> 16)));
    }
    __syncwarp();
  }
}

// Partial records of the merge ("vLLM 深度解析（二）：PagedAttention 核心机制",
// sections 3.2.7 and 3.3: m = max m_j, L = sum l_j e^{m_j - m},
// O = sum O_j l_j e^{m_j - m} / L).  Record (cta, piece, slot) holds, for each
// of the unit's 128 query rows, (m_j, l_j) and the normalised O_j row; O is
// stored as [D / 4][128 rows][4 columns], so that a warp's 16-byte accesses
// to one column group are 512 contiguous bytes and 32 columns of a record
// are one contiguous 16 KB block.  Piece 1 is a unit's first CTA (its tail
// piece), piece 0 any later one.
__device__ __forceinline__ size_t prec(int c, int c0, int b) {
  return (static_cast<size_t>(c) * 2 + (c == c0 ? 1 : 0)) * 2 + b;
}

// The merge of a unit's pieces for one query row (thread i_row of slot b),
// in contributor order c0 .. c1, from the published partials.  Contributor
// `own` (this CTA, merging without publishing) is taken from registers
// (m_ref, l_run) and TMEM (its unnormalised O at tm_o) instead, as the same
// fp32 values it would have published (O_j o_scale / l_j), so the result does not depend on
// which contributor merges; weights and sums are taken in the same order as
// in merge_staged().  Out of line: its registers stay apart from the softmax
// loop's.  Called by every lane of the warp (the TMEM loads are warp-wide).
template <int D>
__device__ __noinline__ void merge_row(const float* __restrict__ part_ml,
                                       const float* __restrict__ part_o, int c0, int c1, int own,
                                       int b, int i_row, float m_ref, float l_run, uint32_t tm_o,
                                       float o_scale, __nv_bfloat16* dst, bool write) {
  const float inv_own = l_run > 0.f ? o_scale / l_run : 0.f;
  auto ml_of = [&](int c) -> float2 {
    return c == own ? make_float2(m_ref, l_run)
                    : __ldcg(reinterpret_cast<const float2*>(part_ml + (prec(c, c0, b) * 128 + i_row) * 2));
  };
  float M = kNegBigP;
  for (int c = c0; c <= c1; c += 4) {
    float2 ml4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) ml4[u] = c + u <= c1 ? ml_of(c + u) : make_float2(kNegBigP, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u) M = fmaxf(M, ml4[u].x);
  }
  float L = 0.f;
  for (int c = c0; c <= c1; c += 4) {
    float2 ml4[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) ml4[u] = c + u <= c1 ? ml_of(c + u) : make_float2(kNegBigP, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (c + u <= c1) L += ml4[u].y * fast_exp2(ml4[u].x - M);
  }
  const float invL = L > 0.f ? 1.f / L : 0.f;
#pragma unroll 1
  for (int cc = 0; cc < D; cc += 16) {
    float mine[16];
    if (own >= 0) {
      tmem_ld16(tm_o + cc, mine);
#pragma unroll
      for (int e = 0; e < 16; ++e) mine[e] *= inv_own;
    }
    float acc[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) acc[e] = 0.f;
    for (int c = c0; c <= c1; c += 2) {
      const bool two = c + 1 <= c1;
      float4 v[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int cu = two ? c + u : c;
        const float4* src = reinterpret_cast<const float4*>(part_o + prec(cu, c0, b) * (D * 128)) +
                            (cc / 4) * 128 + i_row;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          v[u][e] = cu == own ? make_float4(mine[4 * e], mine[4 * e + 1], mine[4 * e + 2], mine[4 * e + 3])
                              : __ldcg(src + e * 128);
      }
      const float2 ml0 = ml_of(c);
      const float2 ml1 = two ? ml_of(c + 1) : make_float2(kNegBigP, 0.f);
      const float w0 = ml0.y * fast_exp2(ml0.x - M);
      const float w1 = ml1.y * fast_exp2(ml1.x - M);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        acc[4 * e] = fmaf(w0, v[0][e].x, acc[4 * e]);
        acc[4 * e + 1] = fmaf(w0, v[0][e].y, acc[4 * e + 1]);
        acc[4 * e + 2] = fmaf(w0, v[0][e].z, acc[4 * e + 2]);
        acc[4 * e + 3] = fmaf(w0, v[0][e].w, acc[4 * e + 3]);
      }
      if (two) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[4 * e] = fmaf(w1, v[1][e].x, acc[4 * e]);
          acc[4 * e + 1] = fmaf(w1, v[1][e].y, acc[4 * e + 1]);
          acc[4 * e + 2] = fmaf(w1, v[1][e].z, acc[4 * e + 2]);
          acc[4 * e + 3] = fmaf(w1, v[1][e].w, acc[4 * e + 3]);
        }
      }
    }
    if (write) {
#pragma unroll
      for (int e = 0; e < 16; e += 8)
        *reinterpret_cast<uint4*>(dst + cc + e) = make_uint4(
            pack_bf16x2(acc[e] * invL, acc[e + 1] * invL), pack_bf16x2(acc[e + 2] * invL, acc[e + 3] * invL),
            pack_bf16x2(acc[e + 4] * invL, acc[e + 5] * invL), pack_bf16x2(acc[e + 6] * invL, acc[e + 7] * invL));
    }
  }
}

// The same merge at a CTA's last segment, with the other contributors'
// records staged in shared memory by bulk copies: their (m, l) records
// first, then their O records 32 columns at a time, up to C::MDATA copies
// in flight, instead of a register round trip per few columns.  Run by the
// 4 warps of slot b (`issuer`: one thread of them issues the copies);
// `area_q` / `area_r`: slot b's free Q buffer and K or V ring.  Returns false
// (error recorded) if a wait ran out; copies already issued are then waited
// for (bounded) before it returns.
template <int D>
__device__ __noinline__ bool merge_staged(const float* __restrict__ part_ml,
                                          const float* __restrict__ part_o, int c0, int c1, int own,
                                          int b, int i_row, bool issuer, float m_ref, float l_run,
                                          uint32_t tm_o, uint32_t area_q, uint32_t area_r,
                                          uint32_t bar_full, uint32_t bar_ml, uint32_t bar_empty,
                                          float o_scale, __nv_bfloat16* dst, bool write,
                                          int32_t* status, int cta) {
  using C = PrefillCfg<D>;
  constexpr int NCH = D / 32;  // 32-column chunks of a record
  const int lane = threadIdx.x & 31;
  const int n_rem = c1 - c0 + 1 - (own >= 0 ? 1 : 0);
  const int total = NCH * n_rem;
  auto buf = [&](int i) -> uint32_t {
    return i < C::MQB ? area_q + i * C::MBUF : area_r + (i - C::MQB) * C::MBUF;
  };
  const uint32_t ml_buf = buf(C::MDATA);
  auto remote = [&](int k) -> int { return c0 + k + (own >= 0 && c0 + k >= own ? 1 : 0); };
  int issued = 0;
  auto issue = [&](int s) {  // copy s: chunk s / n_rem of remote contributor s % n_rem
    const int c = remote(s % n_rem), ch = s / n_rem;
    const uint32_t fb = bar_full + 8 * (s % C::MDATA);
    mbar_arrive_expect_tx(fb, C::MBUF);
    bulk_copy_g2s(buf(s % C::MDATA), part_o + prec(c, c0, b) * (D * 128) + ch * (32 * 128), C::MBUF, fb);
    issued = s + 1;
  };
  if (issuer) {
    // The partials were published (plain stores, a fence, the counter)
    // before the counter this CTA observed; the copies read them through
    // the asynchronous proxy.
    __threadfence();
    fence_proxy_async_global();
    mbar_arrive_expect_tx(bar_ml, n_rem * 1024);
    for (int k = 0; k < n_rem; ++k)
      bulk_copy_g2s(ml_buf + k * 1024, part_ml + prec(remote(k), c0, b) * 256, 1024, bar_ml);
    for (int s = 0; s < min(C::MDATA, total); ++s) issue(s);
  }
  auto wait_all = [&](uint32_t bar, uint32_t parity, int where) -> bool {
    const bool good = __all_sync(0xffffffffu, mbar_wait(bar, parity) ? 1 : 0) != 0;
    if (!good && lane == 0) record_error(status, PA_DEV_WAIT_TIMEOUT, cta, where);
    return good;
  };
  bool ok = wait_all(bar_ml, 0, 86);
  int s = 0;
  if (ok) {
    auto ml_at = [&](int c, int k) -> float2 {
      if (c == own) return make_float2(m_ref, l_run);
      return ld_shared_f2(ml_buf + (k * 128 + i_row) * 8);
    };
    float M = kNegBigP;
    for (int c = c0, k = 0; c <= c1; ++c) {
      M = fmaxf(M, ml_at(c, k).x);
      if (c != own) ++k;
    }
    float L = 0.f;
    for (int c = c0, k = 0; c <= c1; ++c) {
      const float2 ml = ml_at(c, k);
      L += ml.y * fast_exp2(ml.x - M);
      if (c != own) ++k;
    }
    const float invL = L > 0.f ? 1.f / L : 0.f;
    const float inv_own = l_run > 0.f ? o_scale / l_run : 0.f;
#pragma unroll 1
    for (int ch = 0; ch < NCH && ok; ++ch) {
      float acc[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) acc[e] = 0.f;
      for (int c = c0, k = 0; c <= c1 && ok; ++c) {
        const float2 ml = ml_at(c, k);
        const float w = ml.y * fast_exp2(ml.x - M);
        float v[32];
        if (c == own) {
          uint32_t r[32];
          tmem_ld32_async(tm_o + ch * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]) * inv_own;
        } else {
          if (!(ok = wait_all(bar_full + 8 * (s % C::MDATA), (s / C::MDATA) & 1, 87))) break;
          const uint32_t src = buf(s % C::MDATA) + i_row * 16;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint4 u = ld_shared_v4(src + g * 128 * 16);
            v[4 * g] = __uint_as_float(u.x);
            v[4 * g + 1] = __uint_as_float(u.y);
            v[4 * g + 2] = __uint_as_float(u.z);
            v[4 * g + 3] = __uint_as_float(u.w);
          }
          // This warp is done with buffer s; once all four are, it takes copy
          // s + MDATA (only the issuing thread waits for that).
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_empty + 8 * (s % C::MDATA));
          int good = 1;
          if (issuer && s + C::MDATA < total) {
            if (mbar_wait(bar_empty + 8 * (s % C::MDATA), (s / C::MDATA) & 1)) {
              fence_proxy_async_smem();
              issue(s + C::MDATA);
            } else {
              good = 0;
              record_error(status, PA_DEV_WAIT_TIMEOUT, cta, 88);
            }
          }
          if (!(ok = __all_sync(0xffffffffu, good) != 0)) break;
          ++s;
          ++k;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = fmaf(w, v[e], acc[e]);
      }
      if (ok && write) {
#pragma unroll
        for (int e = 0; e < 32; e += 8)
          *reinterpret_cast<uint4*>(dst + ch * 32 + e) = make_uint4(
              pack_bf16x2(acc[e] * invL, acc[e + 1] * invL), pack_bf16x2(acc[e + 2] * invL, acc[e + 3] * invL),
              pack_bf16x2(acc[e + 4] * invL, acc[e + 5] * invL), pack_bf16x2(acc[e + 6] * invL, acc[e + 7] * invL));
      }
    }
  }
  if (!ok && issuer) {
    // No copy may still be landing when the CTA leaves (bounded waits).
    (void)mbar_wait(bar_ml, 0);
    for (int t = max(s, issued - C::MDATA); t < issued; ++t)
      (void)mbar_wait(bar_full + 8 * (t % C::MDATA), (t / C::MDATA) & 1);
  }
  return ok;
}

// KV8: e4m3 K/V cache (k_scale folded into scale_log2, v_scale = o_scale):
// each landed step is converted in place to f16 by its producer warp, each
// slot's Q is converted to f16 (saturating) by the slot's softmax warps, the
// weights are rounded to f16, and the MMAs are f16 x f16 -> fp32.
template <int D, bool KV8>
__global__ void __launch_bounds__(PrefillCfg<D>::THREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
               const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using C = PrefillCfg<D>;
  using B = PBars<C::NST, C::SEGS>;
  constexpr uint32_t IDESC_S = KV8 ? idesc_f16_f32(C::BM, C::BN, 0) : C::IDESC_S;
  constexpr uint32_t IDESC_O = KV8 ? idesc_f16_f32(C::BM, D, 1) : C::IDESC_O;
  const int cta = blockIdx.x;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // swizzle atoms
  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_s = sbase + C::OFF_Q;
  const uint32_t k_s = sbase + C::OFF_K;
  const uint32_t v_s = sbase + C::OFF_V;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int k) -> uint32_t { return bar0 + 8 * k; };
  PSeg* segs = reinterpret_cast<PSeg*>(smem + C::OFF_SEG);
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
  volatile int* fail_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  volatile int* n_k_issued = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 12);
  volatile int* n_v_issued = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  volatile int* n_q_issued = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 20);  // [2]
  volatile int* direct_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 28);

  if (tid == 0) {
    for (int k = 0; k < B::COUNT; ++k) {
      int count = 1;
      if ((k >= B::PFULL && k < B::PFULL + 2) || (k >= B::OFREE && k < B::OFREE + 2)) count = 4;
      if (k >= B::SEGFREE && k < B::SEGFREE + C::SEGS) count = 10;  // MMA, 8 softmax, V producer
      if (k == B::SYNC) count = 8;
      if (k >= B::MEMPTY && k < B::MEMPTY + 10) count = 4;
      if (k >= B::QCONV && k < B::QCONV + 2) count = 4;
      mbar_init(bar(k), count);
    }
    *fail_flag = 0;
    *last_flag = 0;
    *direct_flag = 0;
    *n_k_issued = 0;
    *n_v_issued = 0;
    n_q_issued[0] = 0;
    n_q_issued[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The kernels before this launch (the cache write of this step's tokens)
  // must be complete before anything is read.  Only then may the decode
  // rows of the same call start: they run on the SMs these CTAs leave free.
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  const int GP = (a.group + 1) / 2;        // head pairs per kv head
  const int NP = a.num_kv_heads * GP;      // head pairs (units per query tile)
  auto give_up = [&](int where) {
    record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, where);
    *fail_flag = 1;
  };
  // Cache row of 16-token tile t8 + lane (lane < 8) of request r in the
  // grouped TMA view; an id outside the pool is reported (if `report`) and
  // read as wholly out of bounds (TMA fills zeros).
  auto tile_rows = [&](int r, int t8, int nblk, bool report) -> int {
    const int t16 = t8 + lane;
    if (lane >= 8 || t16 >= nblk) return 0;
    const int id = __ldg(a.block_tables + static_cast<size_t>(r) * a.max_blocks_per_seq + (t16 >> a.tile_shift));
    if (static_cast<unsigned>(id) >= static_cast<unsigned>(a.num_blocks)) {
      if (report) record_error(a.status, PA_DEV_BAD_BLOCK_ID, r, id);
      return a.num_blocks * a.block_size;
    }
    return id * a.block_size + (t16 & ((1 << a.tile_shift) - 1)) * kBlockSize;
  };

  if (warp == 0) {
    // ====================================================== Q / K producer
    if (cta == 0) report_bad_prefill_rows(a, lane);
    const uint64_t policy = l2_policy_evict_first();
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
    }
    // The split is by cost: every key step costs kCostStep and every unit
    // (a segment start: Q load, first S before any softmax, epilogue)
    // another kCostUnit, when every CTA's share is at least one unit start
    // plus one step wide (so that every CTA between a unit's first and last
    // contributor holds one of its steps); else by steps alone.
    // query_start_loc and seq_lens of requests 0 .. REQ_CACHE - 1, copied to
    // shared memory in one round of independent loads.
    int* rq = reinterpret_cast<int*>(smem + C::OFF_REQ);  // [q0 | q1 | seq_len][REQ_CACHE]
    {
      const int nc = min(a.num_seqs, C::REQ_CACHE);
#pragma unroll 1
      for (int r = lane; r < nc; r += 32) {
        rq[r] = __ldg(a.query_start_loc + r);
        rq[C::REQ_CACHE + r] = __ldg(a.query_start_loc + r + 1);
        rq[2 * C::REQ_CACHE + r] = __ldg(a.seq_lens + r);
      }
      __syncwarp();
    }
    auto req_local = [&](int r) -> PReq {
      if (r >= a.num_seqs) return PReq{0, 0, 0, 0, 0};
      if (r >= C::REQ_CACHE) return prefill_req(a, r);
      return make_req(a, rq[r], rq[C::REQ_CACHE + r], rq[2 * C::REQ_CACHE + r]);
    };
    auto req_uniform = req_local;  // every lane reads the same entry
    // (Key steps and units of one head pair fit 32 bits; costs are 64-bit.)
    // With `partition`, also the decode rows' 16-token tiles (per kv head).
    int nsum = 0, usum = 0, dsum = 0;
    const RowLimits lim = row_limits(a);
#pragma unroll 1
    for (int r = lane; r < a.num_seqs; r += 32) {
      int q0, q1, len;
      if (r < C::REQ_CACHE) {
        q0 = rq[r];
        q1 = rq[C::REQ_CACHE + r];
        len = rq[2 * C::REQ_CACHE + r];
      } else {
        q0 = __ldg(a.query_start_loc + r);
        q1 = __ldg(a.query_start_loc + r + 1);
        len = __ldg(a.seq_lens + r);
      }
      const PReq p = tile_req(q0, q1, len, lim);
      nsum += req_steps(p);
      usum += p.ntq;
      if (a.partition) dsum += decode_row_tiles(q0, q1, len, lim);
    }
    nsum = __reduce_add_sync(0xffffffffu, nsum);
    usum = __reduce_add_sync(0xffffffffu, usum);
    const long long Cw = (kCostStep * nsum + kCostUnit * static_cast<long long>(usum)) * NP;
    // The CTAs that work: all, or (mixed batch) the share of the SMs the
    // decode rows leave; the others exit at once.
    const int nct = a.partition
                        ? tile_kernel_sms(Cw, static_cast<long long>(__reduce_add_sync(0xffffffffu, dsum)) *
                                                  a.num_kv_heads,
                                          a.num_ctas, KV8)
                        : a.num_ctas;
    const bool by_cost = nct > 0 && div_ll(Cw, nct) >= kCostStep + kCostUnit;
    const long long CT = by_cost ? kCostStep : 1, CS = by_cost ? kCostUnit : 0;
    const long long Ctot = by_cost ? Cw : static_cast<long long>(nsum) * NP;
    const long long x0 = Ctot > 0 && cta < nct ? range_lo(Ctot, nct, cta) : 0;
    const long long x1 = Ctot > 0 && cta < nct ? range_lo(Ctot, nct, cta + 1) : 0;
    int seg = 0, g = 0;
    int nq[2] = {0, 0};
    bool ok = true;
    auto lane0_wait = [&](uint32_t b, uint32_t parity, int where) -> bool {
      int good = 1;
      if (lane == 0) {
        if (*fail_flag) good = 0;
        else if (!mbar_wait(b, parity)) { give_up(where); good = 0; }
      }
      return __all_sync(0xffffffffu, good) != 0;
    };
    auto seg_slot = [&](int s) -> bool {  // ring slot of segment s is free again
      return s < C::SEGS || lane0_wait(bar(B::SEGFREE + s % C::SEGS), ((s / C::SEGS) - 1) & 1, 60);
    };
    // Steps [j, ..) of a unit whose cost starts at cb: step j starts at
    // cb + CS + CT j.  The first step starting at or after x:
    auto first_step_at = [&](long long cb, long long x) -> long long {
      return x <= cb + CS ? 0 : div_ll(x - cb - CS + CT - 1, CT);
    };
    if (x0 < x1) {
      // The request holding cost position x0, with the key steps and units
      // (of one head pair) of the requests before it.
      int sbase = 0, ubase32 = 0;
      int r = -1;
      // A chunk of 32 requests that ends before x0 is skipped with two warp
      // reductions; inside the one that holds it, inclusive prefixes.
#pragma unroll 1
      for (int rc = 0; rc < a.num_seqs && r < 0; rc += 32) {
        const PReq p = req_local(rc + lane);
        const int st = req_steps(p), nt = p.ntq;
        const int ts = __reduce_add_sync(0xffffffffu, st), tu = __reduce_add_sync(0xffffffffu, nt);
        if ((CT * (sbase + ts) + CS * (ubase32 + tu)) * NP <= x0) {  // past these 32 requests
          sbase += ts;
          ubase32 += tu;
          continue;
        }
        int is = st, iu = nt;
#pragma unroll 1
        for (int o = 1; o < 32; o <<= 1) {
          const int vs = __shfl_up_sync(0xffffffffu, is, o);
          const int vu = __shfl_up_sync(0xffffffffu, iu, o);
          if (lane >= o) {
            is += vs;
            iu += vu;
          }
        }
        // cost up to the end of request rc + lane
        const long long end = (CT * (sbase + is) + CS * (ubase32 + iu)) * NP;
        const int first = __ffs(__ballot_sync(0xffffffffu, end > x0)) - 1;
        sbase += __shfl_sync(0xffffffffu, is - st, first);
        ubase32 += __shfl_sync(0xffffffffu, iu - nt, first);
        r = rc + first;
      }
      const long long base = (CT * sbase + CS * ubase32) * NP;
      const long long ubase = static_cast<long long>(ubase32) * NP;
      // Unit (query tile u, head pair hp) of request r holding x0.
      PReq p = req_uniform(r);
      int u = 0, hp = 0, row0 = 0, rows = 0, kv_end = 0;
      int n_u = unit_steps(p, 0, &row0, &rows, &kv_end);
      long long cb = base;   // cost before the current unit
      long long ub = ubase;  // units before query tile u of request r
      while (cb + NP * (CS + CT * n_u) <= x0) {
        cb += NP * (CS + CT * n_u);
        ++u;
        ub += NP;
        n_u = unit_steps(p, u, &row0, &rows, &kv_end);
      }
      hp = static_cast<int>(div_ll(x0 - cb, CS + CT * n_u));
      cb += hp * (CS + CT * n_u);
      long long j = first_step_at(cb, x0);
      while (ok) {
        if (j >= n_u) {
          // no step of this unit starts in the range: on to the next unit
          cb += CS + CT * n_u;
          j = 0;
          if (++hp == NP) {
            hp = 0;
            ub += NP;
            if (++u == p.ntq) {
              u = 0;
              do {
                p = req_uniform(++r);
              } while (p.ntq == 0 && r < a.num_seqs);
              if (p.ntq == 0) break;  // no more work
            }
          }
          n_u = unit_steps(p, u, &row0, &rows, &kv_end);
        }
        if (cb + CS + CT * j >= x1) break;  // the next step starts past the range
        const int j0 = static_cast<int>(j);
        const int j1 = static_cast<int>(min(static_cast<long long>(n_u), first_step_at(cb, x1)));
        const int kvh = hp / GP;
        const int h0 = kvh * a.group + 2 * (hp % GP);
        const int h1 = 2 * (hp % GP) + 1 < a.group ? h0 + 1 : -1;
        if (!(ok = seg_slot(seg))) break;
        if (lane == 0) {
          PSeg sg;
          sg.r = r;
          sg.q0 = p.q0;
          sg.row0 = row0;
          sg.rows = rows;
          sg.ctx = p.ctx;
          sg.kv_end = kv_end;
          sg.n_kv = n_u;
          sg.j0 = j0;
          sg.j1 = j1;
          sg.h0 = h0;
          sg.h1 = h1;
          sg.kvh = kvh;
          sg.kind = (j0 == 0 && j1 == n_u) ? kSegWhole : (j0 > 0 ? kSegHead : kSegTail);
          sg.unit = static_cast<int>(ub + hp);
          sg.c0 = cta_of_tile(Ctot, nct, cb + CS);
          sg.c1 = cta_of_tile(Ctot, nct, cb + CS + CT * (n_u - 1));
          segs[seg % C::SEGS] = sg;
          mbar_arrive(bar(B::SEGFULL + seg % C::SEGS));
        }
        // Q of both heads (their buffers are free once the previous
        // segment's last S MMA of that slot is done).
        for (int b = 0; b < 2 && ok; ++b) {
          if (b == 1 && h1 < 0) break;
          if (nq[b] > 0 && !(ok = lane0_wait(bar(B::QFREE + b), (nq[b] - 1) & 1, 61))) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(B::QFULL + b), C::QBYTES);
#pragma unroll
            for (int h = 0; h < C::HALVES; ++h)
              tma_load_3d(q_s + b * C::QBYTES + h * C::CHUNK, &qmap, bar(B::QFULL + b), 64 * h,
                          b ? h1 : h0, p.q0 + row0, policy);
            n_q_issued[b] = nq[b] + 1;
          }
          ++nq[b];
        }
        // K of every step: lane L < 8 copies block L of the step.
        const int nblk = (kv_end + kBlockSize - 1) / kBlockSize;
        int rowc = tile_rows(r, j0 * 8, nblk, true);
        if constexpr (KV8) {
          // e4m3: the copy of the segment's next step is issued before this
          // step is waited for and converted (two copies in flight).
          auto issue_raw = [&](int jj, int gg, int row) -> bool {
            const int st = gg % C::NST;
            if (gg >= C::NST && !lane0_wait(bar(B::KFREE + st), ((gg / C::NST) - 1) & 1, 62)) return false;
            const int nb = min(8, nblk - jj * 8);
            if (lane == 0) mbar_arrive_expect_tx(bar(B::KRAW + st), nb * C::RAW_BLOCK);
            __syncwarp();
            if (lane < nb)
              tma_load_3d(k_s + st * C::TBYTES + C::RAW_OFF + lane * C::RAW_BLOCK, &kmap,
                          bar(B::KRAW + st), 0, kvh, row, policy);
            if (lane == 0) *n_k_issued = gg + 1;
            return true;
          };
          if (j0 < j1) ok = issue_raw(j0, g, rowc);
          for (int jj = j0; jj < j1 && ok; ++jj) {
            if (jj + 1 < j1) {
              rowc = tile_rows(r, (jj + 1) * 8, nblk, true);
              if (!(ok = issue_raw(jj + 1, g + 1, rowc))) break;
            }
            const int st = g % C::NST;
            if (!(ok = lane0_wait(bar(B::KRAW + st), (g / C::NST) & 1, 65))) break;
            convert_e4m3_step<D>(k_s + st * C::TBYTES, min(8, nblk - jj * 8), lane);
            fence_proxy_async_smem();  // read by the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B::KFULL + st));
            ++g;
          }
        } else {
          for (int jj = j0; jj < j1 && ok; ++jj) {
            const int st = g % C::NST;
            if (g >= C::NST && !(ok = lane0_wait(bar(B::KFREE + st), ((g / C::NST) - 1) & 1, 62))) break;
            const int nb = min(8, nblk - jj * 8);
            if (lane == 0) mbar_arrive_expect_tx(bar(B::KFULL + st), nb * C::BLOCK_BYTES);
            __syncwarp();
            if (lane < nb)
              tma_load_5d(k_s + st * C::TBYTES + lane * C::BLOCK_BYTES, &kmap, bar(B::KFULL + st), 0,
                          0, 0, rowc / 8, kvh, policy);
            ++g;
            if (lane == 0) *n_k_issued = g;
            if (jj + 1 < j1) rowc = tile_rows(r, (jj + 1) * 8, nblk, true);
          }
        }
        ++seg;
        if (j1 < n_u) break;  // the range ends inside this unit
        j = n_u;              // next unit
      }
    }
    // End record.
    if (ok && (ok = seg_slot(seg)) && lane == 0) {
      segs[seg % C::SEGS].kind = kSegEnd;
      mbar_arrive(bar(B::SEGFULL + seg % C::SEGS));
    }
    if (!ok && lane == 0) *fail_flag = 1;
  } else if (warp == 10) {
    // =========================================================== V producer
    const uint64_t policy = l2_policy_evict_first();
    if (lane == 0) tma_prefetch_desc(&vmap);
    auto warp_wait = [&](uint32_t b, uint32_t parity, int where) -> bool {
      if (*fail_flag) return false;  // one load by the whole warp: the same value
      const bool good = __all_sync(0xffffffffu, mbar_wait(b, parity) ? 1 : 0) != 0;
      if (!good && lane == 0) give_up(where);
      return good;
    };
    bool ok = true;
    int g = 0;
    for (int seg = 0; ok; ++seg) {
      const int slot = seg % C::SEGS;
      if (!(ok = warp_wait(bar(B::SEGFULL + slot), (seg / C::SEGS) & 1, 63))) break;
      const PSeg sg = segs[slot];
      if (sg.kind == kSegEnd) break;
      const int nblk = (sg.kv_end + kBlockSize - 1) / kBlockSize;
      if constexpr (KV8) {
        // As for K: the segment's next step is in flight while this one is
        // converted.
        auto issue_raw = [&](int jj, int gg) -> bool {
          const int st = gg % C::NST;
          const int rowc = tile_rows(sg.r, jj * 8, nblk, false);
          if (gg >= C::NST && !warp_wait(bar(B::VFREE + st), ((gg / C::NST) - 1) & 1, 64)) return false;
          const int nb = min(8, nblk - jj * 8);
          if (lane == 0) mbar_arrive_expect_tx(bar(B::VRAW + st), nb * C::RAW_BLOCK);
          __syncwarp();
          if (lane < nb)
            tma_load_3d(v_s + st * C::TBYTES + C::RAW_OFF + lane * C::RAW_BLOCK, &vmap,
                        bar(B::VRAW + st), 0, sg.kvh, rowc, policy);
          if (lane == 0) *n_v_issued = gg + 1;
          return true;
        };
        if (sg.j0 < sg.j1) ok = issue_raw(sg.j0, g);
        for (int jj = sg.j0; jj < sg.j1 && ok; ++jj) {
          if (jj + 1 < sg.j1 && !(ok = issue_raw(jj + 1, g + 1))) break;
          const int st = g % C::NST;
          if (!(ok = warp_wait(bar(B::VRAW + st), (g / C::NST) & 1, 66))) break;
          convert_e4m3_step<D>(v_s + st * C::TBYTES, min(8, nblk - jj * 8), lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B::VFULL + st));
          ++g;
        }
      } else {
        for (int jj = sg.j0; jj < sg.j1 && ok; ++jj) {
          const int st = g % C::NST;
          const int rowc = tile_rows(sg.r, jj * 8, nblk, false);
          if (g >= C::NST && !(ok = warp_wait(bar(B::VFREE + st), ((g / C::NST) - 1) & 1, 64))) break;
          const int nb = min(8, nblk - jj * 8);
          if (lane == 0) mbar_arrive_expect_tx(bar(B::VFULL + st), nb * C::BLOCK_BYTES);
          __syncwarp();
          if (lane < nb)
            tma_load_5d(v_s + st * C::TBYTES + lane * C::BLOCK_BYTES, &vmap, bar(B::VFULL + st), 0, 0,
                        0, rowc / 8, sg.kvh, policy);
          ++g;
          if (lane == 0) *n_v_issued = g;
        }
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(bar(B::SEGFREE + slot));
    }
    if (!ok && lane == 0) *fail_flag = 1;
  } else if (warp == 1) {
    // ========================================================== MMA issuer
    if (lane == 0) {
      bool ok = true;
      int g = 0, pc[2] = {0, 0}, oc[2] = {0, 0}, qc[2] = {0, 0};
      auto wait = [&](int k, uint32_t parity, int where) -> bool {
        if (*fail_flag) return false;
        if (!mbar_wait(bar(k), parity)) {
          give_up(where);
          return false;
        }
        return true;
      };
      // S_b = Q_b K^T of the K stage st, into TMEM columns 128 b.
      auto issue_s = [&](int b, int st) {
        const uint32_t kst = k_s + st * C::TBYTES;
        const uint32_t qb = q_s + b * C::QBYTES;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t qoff = (ks / 4) * C::CHUNK + (ks % 4) * 32;
          const uint32_t koff = (ks / 4) * 1024 + (ks % 4) * 32;
          umma_bf16(tmem + b * C::BN, sdesc_sw128(qb + qoff, 16, 1024),
                    sdesc_sw128(kst + koff, 16, C::GSTRIDE), IDESC_S, ks > 0);
        }
      };
      // O_b += P_b V of the V stage st (P_b: bf16 in TMEM columns 128 b ..).
      auto issue_pv = [&](int b, int st, bool acc) {
#pragma unroll
        for (int ks = 0; ks < C::BN / 16; ++ks)
          umma_tmem_a(tmem + 256 + b * D, tmem + b * C::BN + ks * 8,
                      sdesc_sw128(v_s + st * C::TBYTES + ks * C::BLOCK_BYTES, 1024, C::GSTRIDE),
                      IDESC_O, (acc || ks > 0) ? 1u : 0u);
      };
      for (int seg = 0; ok; ++seg) {
        const int slot = seg % C::SEGS;
        if (!(ok = wait(B::SEGFULL + slot, (seg / C::SEGS) & 1, 70))) break;
        const PSeg sg = segs[slot];
        if (sg.kind == kSegEnd) break;
        const int n = sg.j1 - sg.j0;
        const int nsl = sg.h1 >= 0 ? 2 : 1;
        for (int b = 0; b < nsl && ok; ++b) ok = wait((KV8 ? B::QCONV : B::QFULL) + b, qc[b]++ & 1, 71);
        ok = ok && wait(B::KFULL + g % C::NST, (g / C::NST) & 1, 72);
        if (!ok) break;
        tc_fence_after();
        for (int b = 0; b < nsl; ++b) {
          issue_s(b, g % C::NST);
          umma_commit(bar(B::SFULL + b));
          if (n == 1) umma_commit(bar(B::QFREE + b));
        }
        umma_commit(bar(B::KFREE + g % C::NST));
        for (int k = 0; k < n && ok; ++k) {
          const int gk = g + k, st = gk % C::NST, st1 = (gk + 1) % C::NST;
          ok = wait(B::VFULL + st, (gk / C::NST) & 1, 73);
          for (int b = 0; b < nsl && ok; ++b) {
            ok = wait(B::PFULL + b, pc[b]++ & 1, 75) &&
                 (k > 0 || oc[b] == 0 || wait(B::OFREE + b, (oc[b] - 1) & 1, 76));
            if (!ok) break;
            tc_fence_after();
            issue_pv(b, st, k > 0);
            if (k + 1 == n) {
              umma_commit(bar(B::OFULL + b));
            } else {
              // S_b of the next step (its K stage may still be landing).
              if (b == 0 && !(ok = wait(B::KFULL + st1, ((gk + 1) / C::NST) & 1, 74))) break;
              tc_fence_after();
              issue_s(b, st1);
              umma_commit(bar(B::SFULL + b));
              if (k + 2 == n) umma_commit(bar(B::QFREE + b));
            }
          }
          if (!ok) break;
          umma_commit(bar(B::VFREE + st));
          if (k + 1 < n) umma_commit(bar(B::KFREE + st1));
        }
        if (!ok) break;
        g += n;
        for (int b = 0; b < nsl; ++b) ++oc[b];
        mbar_arrive(bar(B::SEGFREE + slot));
      }
      if (!ok) *fail_flag = 1;
      // Every MMA issued has completed before TMEM can be released.
      umma_commit(bar(B::DRAIN));
      (void)mbar_wait(bar(B::DRAIN), 0);
    }
    __syncwarp();
  } else {
    // ============================================================ softmax
    // Warps 2-5 serve slot 0, warps 6-9 slot 1; warp w owns TMEM lanes
    // 32 (w % 4) .. + 31, i.e. query row i = 32 (w % 4) + lane of the unit.
    const int b = warp < 6 ? 0 : 1;
    const int i_row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t tm_s = lane_base + b * C::BN;
    const uint32_t tm_o = lane_base + 256 + b * D;
    const float sl2 = a.scale_log2;
    bool ok = true;
    int sc = 0, oc = 0, g = 0, qn = 0;
    uint32_t sync_phase = 0;
    auto all_wait = [&](int k, uint32_t parity, int where) -> bool {
      if (*fail_flag) return false;  // one load by the whole warp: the same value
      const bool good = __all_sync(0xffffffffu, mbar_wait(bar(k), parity) ? 1 : 0) != 0;
      if (!good && lane == 0) give_up(where);
      return good;
    };
    // Barrier of the 8 softmax warps (bounded).
    auto sync8 = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B::SYNC));
      const bool good = all_wait(B::SYNC, sync_phase & 1, 80);
      ++sync_phase;
      return good;
    };
    for (int seg = 0; ok; ++seg) {
      const int slot = seg % C::SEGS;
      if (!(ok = all_wait(B::SEGFULL + slot, (seg / C::SEGS) & 1, 81))) break;
      const volatile PSeg& sg = segs[slot];  // fields read where used (fewer registers)
      if (sg.kind == kSegEnd) break;
      const int n = sg.j1 - sg.j0;
      const bool active = b == 0 || sg.h1 >= 0;
      const int head = b ? sg.h1 : sg.h0;
      const int pslot = sg.kind == kSegTail ? 1 : 0;
      float m_ref = kNegBigP, l_run = 0.f;
      if (KV8 && active) {
        // This slot's Q to f16 in place (same layout), before its first S MMA.
        if (!(ok = all_wait(B::QFULL + b, qn++ & 1, 79))) break;
        const uint32_t qb = q_s + b * C::QBYTES;
        for (int i = (warp & 3) * 32 + lane; i < C::QBYTES / 16; i += 128) {
          const uint4 w = ld_shared_v4(qb + i * 16);
          st_shared_v4(qb + i * 16, make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y),
                                               bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w)));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B::QCONV + b));
      }
      if (active) {
        const int limit = min(sg.ctx + sg.row0 + i_row, sg.kv_end - 1);  // last key this row sees
        for (int k = 0; k < n && ok; ++k) {
          const int key0 = (sg.j0 + k) * C::BN;
          if (!(ok = all_wait(B::SFULL + b, sc++ & 1, 82))) break;
          tc_fence_after();
          const bool masked = key0 + C::BN - 1 > sg.ctx + sg.row0 || key0 + C::BN > sg.kv_end;
          const int nv = limit - key0 + 1;  // visible keys of this row in this step
          // S_b row, half a row (64 columns) at a time; keys past this row's
          // limit get -inf (their weight 2^-inf = 0); only a step on the
          // diagonal or at the end of the keys has any.
          auto load_half = [&](int hf, uint32_t (&sr)[C::BN / 2]) {
            tmem_ld32_async(tm_s + hf * 64, sr);
            tmem_ld32_async(tm_s + hf * 64 + 32, sr + 32);
            tmem_wait_ld();
            if (masked) {
#pragma unroll
              for (int e = 0; e < C::BN / 2; ++e) sr[e] = hf * 64 + e < nv ? sr[e] : 0xff800000u;  // -inf
            }
          };
          float2 ps4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                           make_float2(0.f, 0.f)};
          uint32_t pk[C::BN / 4];
          // Weights of one pair of columns: scale and shift (packed fp32),
          // exponentiate, round to 16 bits for the P.V product; l sums the
          // fp32 weights.
          auto weights = [&](uint32_t s0, uint32_t s1, float m, int e) {
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(s0), __uint_as_float(s1)),
                                        make_float2(sl2, sl2), make_float2(-m, -m));
            const float p0 = fast_exp2(x.x);  // 0 for the masked keys
            const float p1 = fast_exp2(x.y);
            pk[e / 2] = KV8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            ps4[(e / 2) % 4] = __fadd2_rn(ps4[(e / 2) % 4], make_float2(p0, p1));
          };
          // Pass 1: the row maximum; the reference moves (lazily: only when
          // the maximum exceeds it by more than 2^8) before any weight.
          float mx8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t sr[C::BN / 2];
            load_half(hf, sr);
#pragma unroll
            for (int e = 0; e < C::BN / 2; e += 2)
              mx8[(e / 2) % 8] = fmax3(mx8[(e / 2) % 8], __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]));
          }
          const float m_tile = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                     fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) * sl2;
          const bool moved = m_tile > m_ref + kRescaleSlackP;
          float alpha = 1.f;
          if (moved) {
            alpha = fast_exp2(m_ref - m_tile);
            l_run *= alpha;
            m_ref = m_tile;
          }
          const bool rescale = __any_sync(0xffffffffu, moved);
          // Pass 2: the weights; P_b of each half goes over S_b columns that
          // have already been read (P_b: the first half of the S_b columns).
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t sr[C::BN / 2];
            load_half(hf, sr);
#pragma unroll
            for (int e = 0; e < C::BN / 2; e += 2) weights(sr[e], sr[e + 1], m_ref, e);
            tmem_st16_async(tm_s + hf * 32, pk);
            tmem_st16_async(tm_s + hf * 32 + 16, pk + 16);
          }
          const float2 ps = __fadd2_rn(__fadd2_rn(ps4[0], ps4[1]), __fadd2_rn(ps4[2], ps4[3]));
          l_run += ps.x + ps.y;
          if (rescale && k > 0) {  // (warp-uniform: the TMEM accesses are warp-wide)
            // S_b of this step completing means the P_b V before it has
            // completed too: O_b is current and may be rescaled.
#pragma unroll
            for (int c = 0; c < D / 16; ++c) {
              float ov[16];
              tmem_ld16(tm_o + c * 16, ov);
#pragma unroll
              for (int e = 0; e < 16; ++e) ov[e] *= alpha;
              tmem_st16(tm_o + c * 16, ov);
            }
          }
          // V rows of keys past the needed range (or never loaded) may hold
          // NaN: slot 0's warps zero them before the first P.V reads them.
          const int kz = sg.kv_end - key0;  // keys [kz, BN) of this step are unused
          if (b == 0 && kz < C::BN) {
            const int st = (g + k) % C::NST;
            if (!(ok = all_wait(B::VFULL + st, ((g + k) / C::NST) & 1, 83))) break;
            const int nz = (C::BN - kz) * C::HALVES * 8;
            for (int idx = tid - 64; idx < nz; idx += 128) {
              const int row = kz + idx / (C::HALVES * 8);
              const int h = (idx / 8) % C::HALVES;
              st_shared_v4(v_s + st * C::TBYTES + (row >> 4) * C::BLOCK_BYTES + ((row >> 3) & 1) * C::GSTRIDE +
                               h * 1024 + (row & 7) * 128 + (idx % 8) * 16,
                           make_uint4(0u, 0u, 0u, 0u));
            }
            fence_proxy_async_smem();  // the zeroed rows are read by the tensor core
          }
          tmem_wait_st();
          tc_fence_before();  // P_b and O_b writes precede the next MMAs
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B::PFULL + b));
        }
        if (!ok) break;
      }
      if (!ok) break;
      // ---- end of the segment: O_b / l, the partial, or the merge
      const bool whole = sg.kind == kSegWhole;
      const int c0 = sg.c0, c1 = sg.c1;
      const int unit = sg.unit;
      bool direct = false;
      if (!whole) {
        // When every other piece of the unit has already counted, this one
        // is the last: it merges straight from TMEM without publishing.  The
        // unit's first CTA holds its first steps at the end of its range,
        // while every other piece starts its CTA's range (or fills it) and
        // waits for nothing: that CTA alone waits for them, a bounded time
        // (then it publishes like the others).
        if (warp == 2 && lane == 0) {
          int d = 0;
          if (unit < a.max_units) {
            const bool patient = sg.kind == kSegTail;
            const unsigned long long t0 = patient ? global_timer_ns() : 0ull;
            while (true) {
              const unsigned long long cnt = ld_acquire_u64(a.counters + unit);
              if (static_cast<unsigned>(cnt >> 32) == a.epoch &&
                  static_cast<int>(cnt & 0xffffffffu) == c1 - c0) {
                d = 1;
                break;
              }
              if (!patient || global_timer_ns() - t0 > kMergeWaitNs) break;
              __nanosleep(64);
            }
          } else {
            record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, 85);
          }
          *direct_flag = d;
        }
        if (!(ok = sync8())) break;
        direct = *direct_flag != 0;
      }
      if (active) {
        if (!(ok = all_wait(B::OFULL + b, oc++ & 1, 84))) break;
        tc_fence_after();
        if (!direct) {
          const float inv = l_run > 0.f ? a.o_scale / l_run : 0.f;
          const size_t rec = (static_cast<size_t>(cta) * 2 + pslot) * 2 + b;
          __nv_bfloat16* dst_o =
              a.out + (static_cast<size_t>(sg.q0 + sg.row0 + i_row) * a.num_heads + head) * D;
          float4* dst_p = reinterpret_cast<float4*>(a.part_o + rec * (D * 128)) + i_row;
          if (!whole) *reinterpret_cast<float2*>(a.part_ml + (rec * 128 + i_row) * 2) = make_float2(m_ref, l_run);
          // O_b row, 64 columns per TMEM round trip.
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            uint32_t orow[64];
            tmem_ld32_async(tm_o + h * 64, orow);
            tmem_ld32_async(tm_o + h * 64 + 32, orow + 32);
            tmem_wait_ld();
            if (whole) {
              if (i_row < sg.rows) {
#pragma unroll
                for (int e = 0; e < 64; e += 8)
                  *reinterpret_cast<uint4*>(dst_o + h * 64 + e) = make_uint4(
                      pack_bf16x2(__uint_as_float(orow[e]) * inv, __uint_as_float(orow[e + 1]) * inv),
                      pack_bf16x2(__uint_as_float(orow[e + 2]) * inv, __uint_as_float(orow[e + 3]) * inv),
                      pack_bf16x2(__uint_as_float(orow[e + 4]) * inv, __uint_as_float(orow[e + 5]) * inv),
                      pack_bf16x2(__uint_as_float(orow[e + 6]) * inv, __uint_as_float(orow[e + 7]) * inv));
              }
            } else {
#pragma unroll
              for (int e = 0; e < 64; e += 4)
                dst_p[((h * 64 + e) / 4) * C::BM] =
                    make_float4(__uint_as_float(orow[e]) * inv, __uint_as_float(orow[e + 1]) * inv,
                                __uint_as_float(orow[e + 2]) * inv, __uint_as_float(orow[e + 3]) * inv);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B::OFREE + b));
        }
      }
      g += n;
      // Merge: directly (this piece from TMEM), or, after publishing, when
      // this CTA's count completes the unit; one call site for both.
      int own = -2;  // -2: no merge here
      if (!whole && direct) {
        own = cta;
      } else if (!whole) {
        __threadfence();
        if (!(ok = sync8())) break;
        if (warp == 2 && lane == 0)
          *last_flag = unit < a.max_units &&
                               contribute(a.counters + unit, a.epoch, c1 - c0 + 1, a.status, sg.r)
                           ? 1
                           : 0;
        if (!(ok = sync8())) break;
        if (*last_flag) own = -1;
      }
      if (own != -2 && active) {
        __nv_bfloat16* dst =
            a.out + (static_cast<size_t>(sg.q0 + sg.row0 + i_row) * a.num_heads + head) * D;
        if (sg.j1 < sg.n_kv && c1 - c0 + 1 - (own >= 0 ? 1 : 0) <= C::MREM) {
          // The range ends inside this unit, so this is the CTA's last
          // segment: slot b's Q buffer and a K/V ring are free.
          ok = merge_staged<D>(a.part_ml, a.part_o, c0, c1, own, b, i_row, (warp & 3) == 0 && lane == 0,
                               m_ref, l_run, tm_o, q_s + b * C::QBYTES, b ? v_s : k_s,
                               bar(B::MFULL + 5 * b), bar(B::MLFULL + b), bar(B::MEMPTY + 5 * b),
                               a.o_scale, dst, i_row < sg.rows, a.status, cta);
          if (!ok) break;
        } else {
          if (own == -1) __threadfence();
          merge_row<D>(a.part_ml, a.part_o, c0, c1, own, b, i_row, m_ref, l_run, tm_o, a.o_scale,
                       dst, i_row < sg.rows);
        }
      }
      if (active && direct) {  // O_b was read by the merge
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B::OFREE + b));
      }
      if (!whole) {
        if (!(ok = sync8())) break;  // direct_flag and last_flag are read by every warp before they change
        if (warp == 2 && lane == 0 && own != -2) release_pair(a.counters + unit);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B::SEGFREE + slot));
    }
    if (!ok && lane == 0) *fail_flag = 1;
  }

  __syncthreads();
  if (*fail_flag && tid == 0) {
    // Let copies still in flight land before TMEM is released and the CTA
    // leaves (bounded).
    const int nk = *n_k_issued, nv = *n_v_issued;
    const int kb = KV8 ? B::KRAW : B::KFULL, vb = KV8 ? B::VRAW : B::VFULL;
    for (int i = max(0, nk - C::NST); i < nk; ++i)
      (void)mbar_wait(bar(kb + i % C::NST), (i / C::NST) & 1);
    for (int i = max(0, nv - C::NST); i < nv; ++i)
      (void)mbar_wait(bar(vb + i % C::NST), (i / C::NST) & 1);
    for (int b = 0; b < 2; ++b)
      if (n_q_issued[b] > 0) (void)mbar_wait(bar(B::QFULL + b), (n_q_issued[b] - 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool KV8>
cudaError_t launch_prefill_impl(const PrefillArgs& a, const CUtensorMap& qmap,
                                const CUtensorMap& kmap, const CUtensorMap& vmap,
                                cudaStream_t stream) {
  using C = PrefillCfg<D>;
  static bool attr_set[64] = {false};  // per device: set once
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    const cudaError_t err = cudaFuncSetAttribute(prefill_kernel<D, KV8>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  return launch_overlapped(prefill_kernel<D, KV8>, dim3(a.num_ctas), dim3(C::THREADS), C::SMEM,
                           stream, qmap, kmap, vmap, a);
}

}  // namespace

size_t prefill_partials_bytes(int num_ctas, int head_dim) {
  return static_cast<size_t>(num_ctas) * 2 * 2 * 128 * (2 + head_dim) * sizeof(float);
}

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int head_dim, bool kv8, cudaStream_t stream) {
  if (head_dim == 128)
    return kv8 ? launch_prefill_impl<128, true>(a, qmap, kmap, vmap, stream)
               : launch_prefill_impl<128, false>(a, qmap, kmap, vmap, stream);
  if (head_dim == 64)
    return kv8 ? launch_prefill_impl<64, true>(a, qmap, kmap, vmap, stream)
               : launch_prefill_impl<64, false>(a, qmap, kmap, vmap, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
