// prefill.cu -- chunked-prefill attention tiles of a varlen batch on the
// sm_103a tensor cores (tcgen05).
//
// Method ("分块预填充与混合批处理", section 11.6; "vLLM 深度解析（二）：
// PagedAttention 核心机制", sections 2.1, 2.2, 3.1 and 5.2): request r owns
// query rows query_start_loc[r] .. query_start_loc[r+1] - 1; with q_len rows
// and K/V length seq_len, row i sits at position ctx + i (ctx = seq_len -
// q_len) and attends keys 0 .. ctx + i, read through the block table.
// O = softmax(scale * Q K^T) V is computed tile by tile with the online
// softmax state (m, l) per row and never materialises S or P in HBM.
//
// GB300 design.  One CTA owns 128 query rows of one q head of one request
// and is warp-specialised:
//   warps 8, 10 producers: TMA (128-byte swizzle) loads the Q tile once
//               (warp 8) and K (warp 8) and V (warp 10) tiles of 128 keys:
//               eight 16-token blocks gathered through the block table, one
//               copy per block that lands as [8-key group][head_dim half]
//               [8 keys][128 B], a layout both MMAs read directly.  Two-stage
//               rings; a K stage is refilled as soon as its S MMA is done, a
//               V stage as soon as its P.V MMA is done;
//   warp 9      MMA issuer (tcgen05, kind::f16, bf16 in, fp32 accumulate in
//               TMEM):
//                 S_j = Q K_j^T  M = N = 128, K = head_dim, both operands
//                                K-major, into one of two TMEM S buffers;
//                 O  += P_j V_j  M = 128, N = head_dim, K = 128 keys; P_j from
//                                one of two shared-memory buffers (K-major),
//                                V as an MN-major operand exactly as TMA
//                                stored it; O accumulates in TMEM.
//               S_{j+2} is issued as soon as softmax j has S_j in registers
//               and K_{j+2} has landed (before P_j V_j), so the softmax warps
//               find S waiting and run tile after tile without a gap;
//   warps 0-7   softmax: two warps share each 32-row quarter of TMEM and
//               split the key columns (and the columns of O); each reads its
//               part of S_j (tcgen05.ld), applies the causal and length
//               masks, exchanges the row maximum with its partner through two
//               TMEM columns, and writes P_j = exp2(S_j * scale * log2 e - m)
//               as bf16 into the swizzled layout the P.V MMA reads (the
//               scale-and-shift and the row sums two values at a time with
//               packed fp32 instructions; l sums the fp32 weights).
// The reference m of a row moves only when a tile's max exceeds it by more
// than 2^8; then that row of O (in TMEM) and its sum l are rescaled first
// (the final O / l is exact for any reference).  V rows of keys that are out
// of context or were not loaded are zeroed first: they may hold NaN, and a
// zero weight does not cancel a NaN inside the MMA.  Every wait is bounded.
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr float kNegBigP = -1e30f;
constexpr float kRescaleSlackP = 8.0f;  // log2 units

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
  static constexpr int BM = 128;                    // query rows per CTA
  static constexpr int BN = 128;                    // keys per K/V tile (8 blocks)
  static constexpr int HALVES = D / 64;             // 128-byte column chunks of head_dim
  static constexpr int CHUNK = 128 * 128;           // one 128-row x 128-byte swizzled chunk
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + HALVES * CHUNK;         // 2 stages
  static constexpr int OFF_V = OFF_K + 2 * HALVES * CHUNK;     // 2 stages
  static constexpr int OFF_P = OFF_V + 2 * HALVES * CHUNK;     // 2 buffers x 2 key halves
  static constexpr int NBAR = 16;
  static constexpr int OFF_BAR = OFF_P + 4 * CHUNK;
  // Softmax: NSPLIT warps per 32-row TMEM lane quarter, each with 1/NSPLIT
  // of the key columns of S and of the head_dim columns of O.  The parts of
  // a row exchange their maxima (and, at the end, their sums) through TMEM
  // columns XCOL.. (per tile parity) and LCOL.., after S and O.
  static constexpr int NSPLIT = 2;
  static constexpr uint32_t XCOL = 384;
  static constexpr uint32_t LCOL = XCOL + 2 * NSPLIT;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 32 + 1024;            // + 1024-byte alignment slack
  static constexpr int SOFTMAX_WARPS = 4 * NSPLIT;
  static constexpr int THREADS = (SOFTMAX_WARPS + 3) * 32;     // + K producer, MMA issuer, V producer
  static constexpr int HC = BN / NSPLIT;                       // S columns per softmax thread
  static constexpr int HD = D / NSPLIT;                        // O columns per softmax thread
  static_assert(HC % 32 == 0 && HD % 16 == 0 && NSPLIT <= 4, "softmax column split");
  static constexpr uint32_t TMEM_COLS = 512;                   // S0 0, S1 128, O 256
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0);
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 1);
  static constexpr uint32_t BLOCK_BYTES = HALVES * 16 * 128;  // K (or V) of one block
  // K and V blocks land as [8-key group][head_dim half][8 keys][128 B]: the
  // 8-key groups of a tile are GSTRIDE apart, head_dim halves 1 KB apart.
  static constexpr int GSTRIDE = HALVES * 1024;
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// mbarriers (index into the barrier array)
constexpr int kQFull = 0;
constexpr int kKFull = 1;    // [2] K tile landed
constexpr int kVFull = 3;    // [2] V tile landed
constexpr int kKFree = 5;    // [2] S MMA that read the K stage is done
constexpr int kSFull = 7;    // [2] S MMA done
constexpr int kPFull = 9;    // [2] softmax wrote P (and finished reading S)
constexpr int kPVDone = 11;  // [2] P.V MMA done (V stage and P buffer free, O current)
constexpr int kSFree = 13;   // [2] softmax has S in registers (the S buffer may be refilled)
constexpr int kRed = 15;     // softmax-warp barrier (row-max exchange)

// Query tiles of request r (0 for rows that are not prefill rows or whose
// lengths are out of range); each tile is 128 rows of one q head.
__device__ __forceinline__ int prefill_tiles(const PrefillArgs& a, int r) {
  const int q0 = a.query_start_loc[r];
  const int q_len = a.query_start_loc[r + 1] - q0;
  if (q_len <= 1) return 0;
  const int seq_len = a.seq_lens[r];
  if (q_len > seq_len || seq_len > a.max_seq_len || seq_len > a.max_blocks_per_seq * a.block_size ||
      q_len > a.max_query_len || q0 < 0 || q0 + q_len > a.total_q)
    return 0;
  return (q_len + PrefillCfg<64>::BM - 1) / PrefillCfg<64>::BM * a.num_heads;
}

// Reports the prefill rows prefill_tiles() rejects (done once, by CTA 0).
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

// Persistent: CTA c takes tiles c, c + gridDim.x, ... of the batch's tile
// list (requests in order; within a request the last query tile, which
// sees the most keys, first; then the q heads).
template <int D>
__global__ void __launch_bounds__(PrefillCfg<D>::THREADS, 1)
prefill_tile_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using C = PrefillCfg<D>;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // swizzle atoms
  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_s = sbase + C::OFF_Q;
  const uint32_t k_s = sbase + C::OFF_K;
  const uint32_t v_s = sbase + C::OFF_V;
  const uint32_t p_s = sbase + C::OFF_P;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int k) -> uint32_t { return bar0 + 8 * k; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
  volatile int* fail_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* tile_rec = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);  // r, local, found

  if (tid == 0) *fail_flag = 0;
  if (warp == 0) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish();
  }
  // The kernels before this launch (the cache write of this step's tokens)
  // must be complete before anything is read.  Only then may the decode
  // rows of the same call start: they run on the SMs these tiles leave free.
  griddep_wait();
  griddep_launch_dependents();
  if (blockIdx.x == 0 && warp == 1) report_bad_prefill_rows(a, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int scan_r = 0;            // warp 0: first request not yet passed by the tile search
  long long scan_base = 0;   // tiles of the requests before scan_r

  for (long long tile = blockIdx.x;; tile += gridDim.x) {
  // ---- locate the tile (warp 0) and set up this tile's barriers
  if (warp == 0) {
    int r_found = -1;
    long long local = 0;
    for (int rc = scan_r; rc < a.num_seqs && r_found < 0; rc += 32) {
      const int rr = rc + lane;
      const long long nt = rr < a.num_seqs ? prefill_tiles(a, rr) : 0;
      long long incl = nt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, rr < a.num_seqs && scan_base + incl > tile);
      if (hit) {
        const int first = __ffs(hit) - 1;
        const long long excl = __shfl_sync(0xffffffffu, incl - nt, first);
        r_found = rc + first;
        scan_base += excl;
        scan_r = r_found;
        local = tile - scan_base;
      } else {
        scan_base += __shfl_sync(0xffffffffu, incl, 31);
        scan_r = rc + 32;
      }
    }
    if (lane == 0) {
      tile_rec[0] = r_found;
      tile_rec[1] = static_cast<int>(local);
      tile_rec[2] = r_found >= 0 ? 1 : 0;
      for (int k = 0; k <= kRed; ++k) {
        if (tile != blockIdx.x) mbar_inval(bar(k));
        const bool by_softmax = k == kPFull || k == kPFull + 1 || k == kSFree || k == kSFree + 1 ||
                                k == kRed;
        mbar_init(bar(k), by_softmax ? C::SOFTMAX_WARPS : 1);
      }
      fence_mbar_init();
    }
  }
  __syncthreads();
  if (!tile_rec[2]) break;
  const int r = tile_rec[0];
  const int q0 = a.query_start_loc[r];
  const int q_len = a.query_start_loc[r + 1] - q0;
  const int seq_len = a.seq_lens[r];
  const int ntq = (q_len + C::BM - 1) / C::BM;
  const int qt = ntq - 1 - tile_rec[1] / a.num_heads;
  const int head = tile_rec[1] % a.num_heads;
  const int ctx = seq_len - q_len;
  const int row0 = qt * C::BM;                     // first query (within the request)
  const int rows = min(C::BM, q_len - row0);       // valid query rows of this tile
  const int kv_end = ctx + row0 + rows;            // keys [0, kv_end) are needed
  const int n_tiles = (kv_end + C::BN - 1) / C::BN;
  const int nblk_need = (kv_end + kBlockSize - 1) / kBlockSize;
  const int kvh = head / a.group;
  auto give_up = [&](int where) {
    record_error(a.status, PA_DEV_WAIT_TIMEOUT, r, where);
    *fail_flag = 1;
  };

  if (warp == C::SOFTMAX_WARPS || warp == C::SOFTMAX_WARPS + 2) {
    // ===================================================== K and V producers
    // Two warps, so that a K tile is never queued behind the V copy that
    // waits for an earlier P.V MMA.
    const bool is_v = warp != C::SOFTMAX_WARPS;
    const int32_t* bt = a.block_tables + static_cast<size_t>(r) * a.max_blocks_per_seq;
    const uint64_t policy = l2_policy_evict_first();
    auto load_ids = [&](int t) -> int {
      const int b = t * 8 + lane;
      return (lane < 8 && t < n_tiles && b < nblk_need) ? __ldg(bt + (b >> a.tile_shift)) : -1;
    };
    // K or V of tile t into stage t % 2: lane 0 posts the byte count, then
    // lanes 0..7 each issue the TMA copies of their own block (lane b holds
    // the id of block b of the tile).
    auto issue_tile = [&](bool is_v, int t, int ids) {
      const int st = t & 1;
      const int nb = min(8, nblk_need - t * 8);
      const uint32_t full = bar((is_v ? kVFull : kKFull) + st);
      if (lane == 0) mbar_arrive_expect_tx(full, nb * C::BLOCK_BYTES);
      __syncwarp();
      if (lane < nb) {
        // rows 16 (tile mod R) .. + 15 of the block holding tile t * 8 + lane
        int row_c = ids * a.block_size + ((t * 8 + lane) & ((1 << a.tile_shift) - 1)) * kBlockSize;
        if (static_cast<unsigned>(ids) >= static_cast<unsigned>(a.num_blocks)) {
          if (!is_v) record_error(a.status, PA_DEV_BAD_BLOCK_ID, r, ids);
          row_c = a.num_blocks * a.block_size;  // wholly out of bounds: TMA fills zeros
        }
        const uint32_t dst = (is_v ? v_s : k_s) + st * C::HALVES * C::CHUNK + lane * C::BLOCK_BYTES;
        tma_load_5d(dst, is_v ? &vmap : &kmap, full, 0, 0, 0, row_c / 8, kvh, policy);
      }
      __syncwarp();
    };
    if (lane == 0 && is_v) tma_prefetch_desc(&vmap);
    if (lane == 0 && !is_v) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      mbar_arrive_expect_tx(bar(kQFull), C::HALVES * C::CHUNK);
#pragma unroll
      for (int h = 0; h < C::HALVES; ++h)
        tma_load_3d(q_s + h * C::CHUNK, &qmap, bar(kQFull), 64 * h, head, q0 + row0, policy);
    }
    int ids = load_ids(0);
    int ids_next = load_ids(1);
    for (int t = 0; t < n_tiles; ++t) {
      int ok = 1;
      // Stage t % 2 held tile t - 2: a K stage is free once S_{t-2} is done,
      // a V stage once P_{t-2} V_{t-2} is done.
      if (lane == 0 && t >= 2 &&
          !mbar_wait(bar((is_v ? kPVDone : kKFree) + (t & 1)), ((t - 2) >> 1) & 1))
        ok = 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      issue_tile(is_v, t, ids);
      ids = ids_next;
      ids_next = load_ids(t + 2);
    }
  } else if (warp == C::SOFTMAX_WARPS + 1) {
    // ========================================================== MMA issuer
    if (lane == 0) {
      auto issue_s = [&](int t) -> bool {  // S_t = Q K_t^T into S buffer t % 2
        // S buffer t % 2 held S_{t-2}: its softmax must have read it.
        if (t >= 2 && !mbar_wait(bar(kSFree + (t & 1)), ((t - 2) >> 1) & 1)) return false;
        if (!mbar_wait(bar(kKFull + (t & 1)), (t >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t kst = k_s + (t & 1) * C::HALVES * C::CHUNK;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t qoff = (ks / 4) * C::CHUNK + (ks % 4) * 32;
          const uint32_t koff = (ks / 4) * 1024 + (ks % 4) * 32;
          umma_bf16(tmem + (t & 1) * C::BN, sdesc_sw128(q_s + qoff, 16, 1024),
                    sdesc_sw128(kst + koff, 16, C::GSTRIDE), C::IDESC_S, ks > 0);
        }
        umma_commit(bar(kSFull + (t & 1)));
        umma_commit(bar(kKFree + (t & 1)));
        return true;
      };
      bool ok = mbar_wait(bar(kQFull), 0) && issue_s(0) && (n_tiles < 2 || issue_s(1));
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int sb = j & 1;
        // S_{j+2} goes first when its K tile has landed (its S buffer is freed
        // early in softmax j), so the tensor core works while softmax j runs;
        // otherwise P_j V_j goes first and S_{j+2} waits for its K tile.
        bool s_next = j + 2 < n_tiles;
        if (s_next && mbar_wait(bar(kSFree + sb), (j >> 1) & 1) &&
            mbar_try_wait(bar(kKFull + sb), ((j + 2) >> 1) & 1)) {
          ok = issue_s(j + 2);
          s_next = false;
        }
        ok = ok && mbar_wait(bar(kPFull + sb), (j >> 1) & 1) && mbar_wait(bar(kVFull + sb), (j >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < C::BN / 16; ++ks) {
          umma_bf16(tmem + 256, sdesc_sw128(p_s + (sb * 2 + ks / 4) * C::CHUNK + (ks % 4) * 32, 16, 1024),
                    sdesc_sw128(v_s + sb * C::HALVES * C::CHUNK + ks * C::BLOCK_BYTES, 1024, C::GSTRIDE),
                    C::IDESC_O, (j > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(bar(kPVDone + sb));
        if (s_next) ok = issue_s(j + 2);
      }
      if (!ok) give_up(12);
    }
  } else {
    // ============================================================ softmax
    // Warp w serves rows 32 (w % 4) .. + 31 (its TMEM lane quarter) and
    // column part w / 4 of S and of O; thread row i = 32 (w % 4) + lane.
    const int part = warp >> 2;
    const int i_row = (warp & 3) * 32 + lane;
    const uint32_t tmem_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t tmem_o = 256;
    const int limit = min(ctx + row0 + i_row, kv_end - 1);  // last key this row may see
    const float sl2 = a.scale_log2;
    float m_ref = kNegBigP, l_run = 0.f;  // both threads of a row keep the same m_ref
    bool ok = true;
    uint32_t red_phase = 0;
    // Barrier of the softmax warps (bounded; orders the exchange writes).
    auto red_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kRed));
      const int done = mbar_wait(bar(kRed), red_phase & 1) ? 1 : 0;
      ++red_phase;
      return __all_sync(0xffffffffu, done) != 0;
    };
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + sb), (j >> 1) & 1) ? 1 : 0) != 0;
      if (!ok) break;
      tc_fence_after();
      uint32_t sraw[C::HC];
#pragma unroll
      for (int c = 0; c < C::HC / 32; ++c)
        tmem_ld32_async(tmem_row + sb * C::BN + part * C::HC + c * 32, sraw + 32 * c);
      tmem_wait_ld();
      tc_fence_before();  // S_j is in registers: the S MMA of tile j + 2 may overwrite it
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kSFree + sb));
      const int key0 = j * C::BN + part * C::HC;  // key of this thread's first column
      const bool full_tile = j * C::BN + C::BN - 1 <= ctx + row0 && j * C::BN + C::BN <= seq_len;
      float mx8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx8[u] = -INFINITY;
      if (full_tile) {
#pragma unroll
        for (int e = 0; e < C::HC; e += 2)
          mx8[(e / 2) % 8] = fmax3(mx8[(e / 2) % 8], __uint_as_float(sraw[e]), __uint_as_float(sraw[e + 1]));
      } else {
#pragma unroll
        for (int e = 0; e < C::HC; e += 2)
          mx8[(e / 2) % 8] = fmax3(mx8[(e / 2) % 8],
                                   key0 + e <= limit ? __uint_as_float(sraw[e]) : -INFINITY,
                                   key0 + e + 1 <= limit ? __uint_as_float(sraw[e + 1]) : -INFINITY);
      }
      float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                       fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      // The row's maximum over all parts (TMEM columns of this tile parity).
      const uint32_t xcol = tmem_row + C::XCOL + sb * C::NSPLIT;
      tmem_st1(xcol + part, mx);
      tc_fence_before();
      if (!(ok = red_sync())) break;
      tc_fence_after();
      {
        float xv[4];
        tmem_ld4(xcol, xv);
#pragma unroll
        for (int p2 = 0; p2 < C::NSPLIT; ++p2) mx = fmaxf(mx, xv[p2]);
      }
      const float m_tile = mx * sl2;
      const bool need = m_tile > m_ref + kRescaleSlackP;
      if (__any_sync(0xffffffffu, need)) {
        // O (in TMEM) must hold P_{j-1} V_{j-1} before its rows are rescaled.
        if (j > 0)
          ok = __all_sync(0xffffffffu,
                          mbar_wait(bar(kPVDone + ((j - 1) & 1)), ((j - 1) >> 1) & 1) ? 1 : 0) != 0;
        if (!ok) break;
        tc_fence_after();
        const float m_new = need ? m_tile : m_ref;
        const float alpha = fast_exp2(m_ref - m_new);
        if (j > 0) {
#pragma unroll
          for (int c = 0; c < C::HD / 16; ++c) {
            float ov[16];
            tmem_ld16(tmem_row + tmem_o + part * C::HD + c * 16, ov);
#pragma unroll
            for (int e = 0; e < 16; ++e) ov[e] *= alpha;
            tmem_st16(tmem_row + tmem_o + part * C::HD + c * 16, ov);
          }
        }
        l_run *= alpha;
        m_ref = m_new;
      }
      // P buffer sb was read by P_{j-2} V_{j-2}: it must be done.
      if (j >= 2)
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kPVDone + sb), ((j - 2) >> 1) & 1) ? 1 : 0) != 0;
      if (!ok) break;
      // Weights: scale and shift two at a time (packed fp32), exponentiate,
      // round to bf16 for the P.V product; l sums the fp32 weights.
      float2 ps4[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) ps4[u] = make_float2(0.f, 0.f);
      const float2 sl2v = make_float2(sl2, sl2), mneg = make_float2(-m_ref, -m_ref);
#pragma unroll
      for (int c = 0; c < C::HC / 32; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int k = c * 32 + e;
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(sraw[k]), __uint_as_float(sraw[k + 1])),
                                      sl2v, mneg);
          float p0 = fast_exp2(x.x);
          float p1 = fast_exp2(x.y);
          if (!full_tile) {
            p0 = key0 + k <= limit ? p0 : 0.f;
            p1 = key0 + k + 1 <= limit ? p1 : 0.f;
          }
          pk[e / 2] = pack_bf16x2(p0, p1);
          ps4[(e / 2) % 4] = __fadd2_rn(ps4[(e / 2) % 4], make_float2(p0, p1));
        }
        // keys part*HC + c*32 .. +31: 16-byte chunks cb .. cb + 3 of key half kh
        const int kfirst = part * C::HC + c * 32;
        const int kh = kfirst >> 6, cb = (kfirst & 63) >> 3;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = cb + q;
          const uint32_t addr =
              p_s + (sb * 2 + kh) * C::CHUNK + i_row * 128 + ((chunk ^ (i_row & 7)) * 16);
          st_shared_v4(addr, make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]));
        }
      }
      const float2 ps01 = __fadd2_rn(ps4[0], ps4[1]), ps23 = __fadd2_rn(ps4[2], ps4[3]);
      const float2 ps = __fadd2_rn(ps01, ps23);
      l_run += ps.x + ps.y;
      // V rows of keys past the needed range or never loaded may hold NaN.
      const int kz = kv_end - j * C::BN;  // keys [kz, BN) of this tile are unused
      if (kz < C::BN) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(kVFull + sb), (j >> 1) & 1) ? 1 : 0) != 0;
        if (!ok) break;
        const int nz = (C::BN - max(kz, 0)) * C::HALVES * 8;
        for (int idx = tid; idx < nz; idx += C::SOFTMAX_WARPS * 32) {
          const int row = max(kz, 0) + idx / (C::HALVES * 8);
          const int h = (idx / 8) % C::HALVES;
          st_shared_v4(v_s + sb * C::HALVES * C::CHUNK + (row >> 4) * C::BLOCK_BYTES +
                           ((row >> 3) & 1) * C::GSTRIDE + h * 1024 + (row & 7) * 128 + (idx % 8) * 16,
                       make_uint4(0u, 0u, 0u, 0u));
        }
      }
      fence_proxy_async_smem();  // P_j and the zeroed rows are read by the tensor core
      tc_fence_before();         // S_j reads and O rescales precede the next MMAs
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kPFull + sb));
    }
    // ---- epilogue: O / l
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(kPVDone + ((n_tiles - 1) & 1)),
                                             ((n_tiles - 1) >> 1) & 1) ? 1 : 0) != 0;
    if (ok) {
      tc_fence_after();
      tmem_st1(tmem_row + C::LCOL + part, l_run);
      tc_fence_before();
      ok = red_sync();
    }
    if (ok) {
      tc_fence_after();
      float lv[4];
      tmem_ld4(tmem_row + C::LCOL, lv);
      float lsum = 0.f;
#pragma unroll
      for (int p2 = 0; p2 < C::NSPLIT; ++p2) lsum += lv[p2];
      const float inv = 1.f / lsum;
      __nv_bfloat16* dst =
          a.out + (static_cast<size_t>(q0 + row0 + i_row) * a.num_heads + head) * D + part * C::HD;
#pragma unroll
      for (int c = 0; c < C::HD / 16; ++c) {
        float ov[16];
        tmem_ld16(tmem_row + tmem_o + part * C::HD + c * 16, ov);
        if (i_row < rows) {
#pragma unroll
          for (int e = 0; e < 16; e += 8) {
            const uint4 v = make_uint4(pack_bf16x2(ov[e] * inv, ov[e + 1] * inv),
                                       pack_bf16x2(ov[e + 2] * inv, ov[e + 3] * inv),
                                       pack_bf16x2(ov[e + 4] * inv, ov[e + 5] * inv),
                                       pack_bf16x2(ov[e + 6] * inv, ov[e + 7] * inv));
            *reinterpret_cast<uint4*>(dst + c * 16 + e) = v;
          }
        }
      }
    } else if (lane == 0) {
      give_up(13);
    }
  }

  __syncthreads();  // end of the tile: every copy and MMA of it has completed
  if (*fail_flag) {
    if (tid == 0) {
      // Let copies and MMAs still in flight finish before TMEM is released
      // and the CTA leaves (bounded; some of these phases may never come).
      for (int k = 0; k < kRed; ++k) (void)mbar_wait(bar(k), 0);
    }
    break;
  }
  }  // tiles

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
cudaError_t launch_prefill_impl(const PrefillArgs& a, const CUtensorMap& qmap,
                                const CUtensorMap& kmap, const CUtensorMap& vmap,
                                cudaStream_t stream) {
  using C = PrefillCfg<D>;
  cudaError_t err = cudaFuncSetAttribute(prefill_tile_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  return launch_overlapped(prefill_tile_kernel<D>, dim3(a.num_ctas), dim3(C::THREADS), C::SMEM,
                           stream, qmap, kmap, vmap, a);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int head_dim, cudaStream_t stream) {
  if (head_dim == 128) return launch_prefill_impl<128>(a, qmap, kmap, vmap, stream);
  if (head_dim == 64) return launch_prefill_impl<64>(a, qmap, kmap, vmap, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
