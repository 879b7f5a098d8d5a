// decode_tc.cu -- paged decode attention on the sm_103a tensor cores.
//
// Method ("vLLM 深度解析（二）：PagedAttention 核心机制"):
//   section 3.1  a request's token t lives in physical block
//                block_table[r][t / 16] at offset t % 16;
//   section 2.2  online softmax: a running (m, l, A) per query row, merged
//                chunk by chunk, O = A / l at the end;
//   section 3.2  scores of tokens >= seq_len are excluded and the V rows of
//                out-of-context slots are zeroed before they are used;
//   sections 3.2.7, 3.3  pieces of a long context are merged through their
//                (m_j, l_j, O_j) (decode_common.cuh).
//
// GB300 design.  The decode of one (request, kv head) pair is two skinny
// matrix products per 128-token chunk, with the G <= 16 q heads of the kv
// head as the narrow dimension:
//   S^T = K Q^T     M = 128 tokens, N = 16 (G heads, padded), K = head_dim;
//                   A = the K chunk (K-major, 128-byte swizzle), B = q;
//   O^T += V^T P^T  M = head_dim (128; at head_dim 64 the upper half of the
//                   product is unused), N = 16, K = 128 tokens;
//                   A = the V chunk read MN-major, B = P^T (K-major).
// Both accumulate in TMEM (fp32); the tensor core does all the FMAs, so the
// CUDA cores only run the softmax (a few exp2 per token) and the kernel's
// time is the K/V stream.  One CTA per SM keeps up to three 64 KB chunks of
// K and V in flight.  Each (block, kv head) of K and of V is one 4 KB TMA
// copy of a 5-D box that lands as [8-token group][head_dim half][8 tokens]
// [128 B], 128-byte swizzled: the 8-token groups of a chunk then sit at one
// stride, a layout both MMAs read as it is (the SM's TMA unit handles a
// roughly fixed number of copies per microsecond, so fewer, larger copies
// mean more bytes in flight).  A chunk's K stage is refilled as soon as its
// S MMA is done, its V stage as soon as its P.V MMA is done.
//
// Warp roles (352 threads):
//   warp 0      K producer: walks this CTA's range of whole 128-token
//               chunks (a split by cost: see kCostSeg),
//               writes one record per segment (the run of one pair's blocks
//               in the range), loads that segment's q and the K of every
//               chunk of 8 blocks, and leaves a record per chunk (block rows,
//               kv head) for the V producer;
//   warp 10     V producer: the V of every chunk, so that issuing K and V
//               copies overlaps;
//   warp 1      MMA issuer: S(j), then P.V(j - 1), chunk after chunk;
//   warps 2-5   softmax: thread i owns token i of the chunk (TMEM lane i).
//               Per head, each warp takes the maximum of its 32 scores with
//               one redux.sync on order-preserving integer keys; the four
//               warps exchange those through shared memory.  The reference
//               max moves only when it is exceeded by more than 2^8, and
//               then O^T (in TMEM) and l are rescaled first.  At the end of
//               a segment the warps publish m and their partial sums of l
//               and go straight on with the next segment;
//   warps 6-9   epilogue: thread i owns row i (head_dim index) of O^T; per
//               segment it waits for the last P.V, divides by l and writes
//               the bf16 output, or writes a partial and, if it is the last
//               contributor of the pair, merges the partials.
// Every wait is bounded; a timeout records PA_DEV_WAIT_TIMEOUT.
#include "decode_common.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr float kNegBigTc = -1e30f;
constexpr float kSlackTc = 8.0f;  // log2 units
constexpr int kEndSeg = 7;        // segment record kind: no more work

template <int D, int GM, bool KV8 = false>
struct TcCfg {
  static constexpr int HALVES = D / 64;             // 128-byte column chunks of head_dim
  static constexpr int CB = 8;                      // blocks per chunk
  static constexpr int CT = CB * kBlockSize;        // tokens per chunk (MMA M)
  static constexpr int N = 16;                      // MMA N: the group's q heads, padded
  static constexpr int BLK = HALVES * kBlockSize * 128;  // 16-bit K (or V) bytes of one block
  static constexpr int BLK8 = kBlockSize * D;       // e4m3 K (or V) bytes of one block
  // A 16-bit block is [8-token group][head_dim half][8 tokens][128 B]: the
  // 8-token groups of a chunk are GSTRIDE apart, head_dim halves 1 KB apart.
  static constexpr int GSTRIDE = HALVES * 1024;
  static constexpr int STAGE = CB * BLK;            // one 16-bit chunk of K (or of V)
  static constexpr int RSTAGE = KV8 ? CB * BLK8 : STAGE;  // one chunk as it lands
  // K stages = V stages (as they land; an e4m3 stage is half as large).
  static constexpr int NST = KV8 ? (D == 128 ? 4 : 8) : (D == 128 ? 3 : 6);
  // e4m3: converted chunks, K (f16) in TMEM and V (f16) in shared memory.
  static constexpr int NCK = KV8 ? 3 : 0;
  static constexpr int NCV = KV8 ? 2 : 0;
  static constexpr int SLOTS = 4;                   // segment records / q buffers
  static constexpr int QSLOT = HALVES * N * 128;    // q of a segment: [half][16 rows][128 B]
  static constexpr int PBUF = 2 * N * 128;          // P^T: [token half][16 rows][128 B]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NST * RSTAGE;
  static constexpr int OFF_VC = OFF_V + NST * RSTAGE;  // converted V (e4m3 caches)
  static constexpr int OFF_Q = OFF_VC + NCV * STAGE;  // also absorbs the unused half of A at D = 64
  static constexpr int OFF_P = OFF_Q + SLOTS * QSLOT;
  static constexpr int OFF_SEG = OFF_P + 2 * PBUF;
  static constexpr int SEG_BYTES = 48;
  static constexpr int OFF_RED = OFF_SEG + SLOTS * SEG_BYTES;  // [2][4][GM] max keys
  static constexpr int OFF_ML = OFF_RED + 2 * 4 * GM * 4;       // [SLOTS][5][GM]: m, 4 partial l
  static constexpr int NREC = 2 * NST;              // chunk records (K producer -> V producer)
  static constexpr int OFF_REC = OFF_ML + SLOTS * 5 * GM * 4;  // [NREC][12] ints
  static constexpr int OFF_BAR = OFF_REC + NREC * 48;
  static constexpr int NBAR = 4 * NST + 3 * SLOTS + 2 * 6 + 2 + NREC + 2 * NCK + 2 * NCV + SLOTS;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;  // + 1024-byte alignment slack
  static constexpr int THREADS = (KV8 ? 15 : 11) * 32;  // + 4 converter warps for e4m3
  // TMEM: S0 0, S1 16, O0 32, O1 48; e4m3: converted K chunks from KCOL.
  static constexpr uint32_t KCOL = 64;
  static constexpr uint32_t TMEM_COLS = KV8 ? 256 : 64;
  static constexpr uint32_t IDESC_S = KV8 ? idesc_f16_f32(CT, N, 0, 0) : idesc_bf16_f32(CT, N, 0, 0);
  static constexpr uint32_t IDESC_O = KV8 ? idesc_f16_f32(128, N, 0, 1) : idesc_bf16_f32(128, N, 0, 1);
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(GM == 4 || GM == 8 || GM == 16, "group bucket");
  static_assert(KCOL + NCK * (D / 2) <= TMEM_COLS, "tensor memory");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// Barrier indices.
template <int NST, int SLOTS, int NREC, int NCK, int NCV>
struct TcBars {
  static constexpr int KFULL = 0;                 // [NST] K chunk landed
  static constexpr int KFREE = KFULL + NST;       // [NST] S MMA (e4m3: the converter) done with it
  static constexpr int VFULL = KFREE + NST;       // [NST]
  static constexpr int VFREE = VFULL + NST;       // [NST] P.V MMA (e4m3: the converter) done with it
  static constexpr int QFULL = VFREE + NST;       // [SLOTS] segment record + q landed
  static constexpr int LREADY = QFULL + SLOTS;    // [SLOTS] softmax published m, l (4 warps)
  static constexpr int SEGFREE = LREADY + SLOTS;  // [SLOTS] epilogue done with the slot (4 warps)
  static constexpr int SFULL = SEGFREE + SLOTS;   // [2] S^T in TMEM
  static constexpr int SFREE = SFULL + 2;         // [2] softmax read S^T (4 warps)
  static constexpr int PFULL = SFREE + 2;         // [2] P^T written (4 warps)
  static constexpr int PVDONE = PFULL + 2;        // [2] P.V MMA done
  static constexpr int OFULL = PVDONE + 2;        // [2] last P.V of a segment done
  static constexpr int OFREE = OFULL + 2;         // [2] epilogue read O^T (4 warps)
  static constexpr int RED = OFREE + 2;           // softmax-warp barrier (4 warps)
  static constexpr int ERED = RED + 1;            // epilogue-warp barrier (4 warps)
  static constexpr int CREC = ERED + 1;           // [NREC] chunk record written
  static constexpr int KCFULL = CREC + NREC;      // [NCK] converted K in TMEM (4 converter warps)
  static constexpr int KCFREE = KCFULL + NCK;     // [NCK] S MMA done reading it
  static constexpr int VCFULL = KCFREE + NCK;     // [NCV] converted V (4 converter warps)
  static constexpr int VCFREE = VCFULL + NCV;     // [NCV] P.V MMA done reading it
  static constexpr int QCONV = VCFREE + NCV;      // [SLOTS] q converted to f16 (4 converter warps)
  static constexpr int COUNT = QCONV + SLOTS;
};

// A segment: the run of 16-token tiles [b0, b0 + nseg) of one (request, kv
// head) pair inside this CTA's range.  This kernel splits the batch in
// units of whole 128-token chunks (8 tiles), so a range boundary never cuts
// a chunk: only the last chunk of a pair can be partial.
struct TcSeg {
  int row;       // q / out row of the request
  int seq_len;
  int npair;     // chunks of the (request, kv head) pair (the split's unit)
  int b0;
  int nseg;
  int kind;      // kWhole, kHead, kTail or kEndSeg
  int r;
  int kvh;
  long long t0;  // number of the pair's first chunk
  long long c0;  // split cost at which the pair's first chunk starts (see kCostSeg)
};
static_assert(sizeof(TcSeg) <= 48, "segment record");

// The batch's chunks are split over the CTAs by cost, not by count: every
// chunk costs kCostChunk and every (request, kv head) segment another
// kCostSeg.  A segment start (q load, first S before any softmax, partial
// last chunk, hand-off) costs about two chunks: on the 70B-shaped
// shared-prefix batch with equal chunk counts a CTA took 216 us + 1.84 us
// per segment of its range (R^2 0.92, 3 to 42 segments per CTA), and the
// decode took 286.8 / 268 / 256 / 254 / 261 us with kCostSeg = 0 / 8 / 13 /
// 18 / 24.
constexpr int kCostChunk = 8;
constexpr int kCostSeg = 16;

// Order-preserving map between fp32 and int32 (its own inverse): signed
// integer comparison of the keys orders the floats (NaN excepted).
__device__ __forceinline__ int f2key(float x) {
  const int b = __float_as_int(x);
  return b >= 0 ? b : (b ^ 0x7fffffff);
}
__device__ __forceinline__ float key2f(int k) { return __int_as_float(k >= 0 ? k : (k ^ 0x7fffffff)); }

// ---- e4m3 caches: every e4m3 value is exact in f16, so the converter warps
// turn the landed K and V bytes into f16 operands without rounding; q and
// the weights are rounded to f16 (q saturates at +-65504).
// 16-byte chunk c of token row t of a landed e4m3 block (16 rows of head_dim
// bytes, 128-byte swizzle at head_dim 128, 64-byte at 64).
template <int D>
__device__ __forceinline__ uint32_t e8_chunk(int t, int c) {
  const int sw = D == 128 ? (t & 7) : ((t >> 1) & 3);
  return static_cast<uint32_t>(t * D + ((c ^ sw) * 16));
}

template <int D, int GM, bool KV8>
__global__ void __launch_bounds__(TcCfg<D, GM, KV8>::THREADS, 1)
paged_decode_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  using C = TcCfg<D, GM, KV8>;
  using B = TcBars<C::NST, C::SLOTS, C::NREC, C::NCK, C::NCV>;
  const int cta = blockIdx.x;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // swizzle atoms
  const uint32_t sbase = smem_u32(smem);
  const uint32_t k_s = sbase + C::OFF_K;
  const uint32_t v_s = sbase + C::OFF_V;
  const uint32_t vc_s = sbase + C::OFF_VC;  // e4m3 caches: V converted to f16
  const uint32_t q_s = sbase + C::OFF_Q;
  const uint32_t p_s = sbase + C::OFF_P;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int k) -> uint32_t { return bar0 + 8 * k; };
  TcSeg* segs = reinterpret_cast<TcSeg*>(smem + C::OFF_SEG);
  int* red_key = reinterpret_cast<int*>(smem + C::OFF_RED);    // [2][4][GM]
  float* seg_ml = reinterpret_cast<float*>(smem + C::OFF_ML);  // [SLOTS][5][GM]
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);
  volatile int* fail_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);
  volatile int* n_chunks_issued = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 12);
  volatile int* n_s_issued = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  volatile int* n_pv_issued = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 20);
  volatile long long* total_tiles = reinterpret_cast<volatile long long*>(smem + C::OFF_MISC + 24);
  volatile int* n_segs_issued = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 32);
  volatile int* n_v_issued = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 36);
  volatile long long* total_cost = reinterpret_cast<volatile long long*>(smem + C::OFF_MISC + 40);
  volatile int* cost_chunk = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 48);
  // [NREC][12]: V rows of 8 blocks, kv head, blocks, valid tokens, first chunk of segment slot + 1
  int* recs = reinterpret_cast<int*>(smem + C::OFF_REC);

  if (tid == 0) {
    for (int k = 0; k < B::COUNT; ++k) {
      const bool four = (k >= B::LREADY && k < B::SEGFREE + C::SLOTS) ||
                        (k >= B::SFREE && k < B::SFREE + 2) || (k >= B::PFULL && k < B::PFULL + 2) ||
                        (k >= B::OFREE && k < B::OFREE + 2) || k == B::RED || k == B::ERED ||
                        // e4m3: the converter warps free the landed stages and fill
                        // the converted K, V and q
                        (KV8 && ((k >= B::KFREE && k < B::KFREE + C::NST) ||
                                 (k >= B::VFREE && k < B::VFREE + C::NST) ||
                                 (k >= B::KCFULL && k < B::KCFULL + C::NCK) ||
                                 (k >= B::VCFULL && k < B::VCFULL + C::NCV) ||
                                 (k >= B::QCONV && k < B::QCONV + C::SLOTS)));
      mbar_init(bar(k), four ? 4 : 1);
    }
    *fail_flag = 0;
    *last_flag = 0;
    *n_chunks_issued = 0;
    *n_s_issued = 0;
    *n_pv_issued = 0;
    *n_segs_issued = 0;
    *n_v_issued = 0;
    *total_tiles = 0;
    *total_cost = 0;
    *cost_chunk = 1;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!a.defer_griddep) griddep_wait();  // the cache write before this launch may still be finishing
  const uint32_t tmem = *tmem_slot;
  auto give_up = [&](int where) {
    record_error(a.status, PA_DEV_WAIT_TIMEOUT, cta, where);
    *fail_flag = 1;
  };

  if (warp == 0) {
    // ============================================================ producer
    if (cta == 0) report_bad_rows(a, lane);
    // Block counts, lengths and q rows of requests 0 .. 32 kReqCache - 1 stay
    // in registers (lane L holds requests 32 k + L); one pass of independent
    // loads gives the batch's tile total.
    constexpr int kReqCache = 8;
    int c_nb[kReqCache], c_len[kReqCache], c_row[kReqCache];
    long long nb_sum = 0, nreq = 0;  // chunks per kv head; requests with chunks
#pragma unroll
    for (int k = 0; k < kReqCache; ++k) {
      const int r = 32 * k + lane;
      c_nb[k] = 0;
      c_len[k] = 0;
      c_row[k] = 0;
      int lv = 0, rv = 0;
      if (r < a.num_seqs) c_nb[k] = request_blocks(a, r, &lv, &rv);
      c_len[k] = lv;
      c_row[k] = rv;
      nb_sum += (c_nb[k] + C::CB - 1) / C::CB;  // chunks
      nreq += c_nb[k] > 0 ? 1 : 0;
    }
    for (int r = 32 * kReqCache + lane; r < a.num_seqs; r += 32) {
      int len, row;
      const int nbv = request_blocks(a, r, &len, &row);
      nb_sum += (nbv + C::CB - 1) / C::CB;
      nreq += nbv > 0 ? 1 : 0;
    }
    nb_sum = warp_sum_ll(nb_sum);  // warp reductions: far faster than shuffle chains here
    nreq = warp_sum_ll(nreq);
    const long long W = nb_sum * a.num_kv_heads;
    // Split by cost when every CTA's share spans at least one whole gap
    // between chunk starts (so no CTA's range is empty); else by chunks.
    const long long Cw = a.num_kv_heads * (kCostChunk * nb_sum + kCostSeg * nreq);
    const bool by_cost = W > 0 && Cw / a.num_ctas >= kCostChunk + kCostSeg;
    const int cu_chunk = by_cost ? kCostChunk : 1;
    const int cu_seg = by_cost ? kCostSeg : 0;
    const long long Ctot = by_cost ? Cw : W;
    // (blocks) -> chunks of a request (every lane); cached for the first
    // 32 kReqCache requests.
    auto req_nb = [&](int r) -> int {
      int nbv = 0;
      if (r < 32 * kReqCache) {
#pragma unroll
        for (int m = 0; m < kReqCache; ++m)
          if (m == (r >> 5)) nbv = c_nb[m];
        nbv = __shfl_sync(0xffffffffu, nbv, r & 31);
      } else if (r < a.num_seqs) {
        int lv, rv;
        nbv = request_blocks(a, r, &lv, &rv);
      }
      return nbv;
    };
    // The first chunk whose cost start is >= x (whole warp): the chunk u of
    // (request r, kv head h, chunk j) starts at cost_base(r) + h (cu_chunk
    // nc_r + cu_seg) + cu_seg + cu_chunk j.
    auto chunk_at_cost = [&](long long x) -> long long {
      long long cb = 0, chb = 0;
      for (int rc = 0; rc < a.num_seqs; rc += 32) {
        const int r = rc + lane;
        const int nc = (req_nb(r) + C::CB - 1) / C::CB;
        const long long ct = nc > 0 ? a.num_kv_heads * (static_cast<long long>(cu_chunk) * nc + cu_seg) : 0;
        const long long nt = static_cast<long long>(nc) * a.num_kv_heads;
        const long long tct = warp_sum_ll(ct);
        if (cb + tct <= x) {  // x lies past these 32 requests
          cb += tct;
          chb += warp_sum_ll(nt);
          continue;
        }
        long long ic = ct, in = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long vc = __shfl_up_sync(0xffffffffu, ic, o);
          const long long vn = __shfl_up_sync(0xffffffffu, in, o);
          if (lane >= o) {
            ic += vc;
            in += vn;
          }
        }
        const unsigned hit = __ballot_sync(0xffffffffu, r < a.num_seqs && cb + ic > x);
        if (hit) {
          const int first = __ffs(hit) - 1;
          const long long cbr = cb + __shfl_sync(0xffffffffu, ic - ct, first);
          const long long chr = chb + __shfl_sync(0xffffffffu, in - nt, first);
          const int ncr = __shfl_sync(0xffffffffu, nc, first);
          const long long segcost = static_cast<long long>(cu_chunk) * ncr + cu_seg;
          const long long off = x - cbr;
          const long long h = off / segcost, o = off % segcost;
          const long long j = o <= cu_seg ? 0 : (o - cu_seg + cu_chunk - 1) / cu_chunk;
          return chr + h * ncr + j;
        }
        cb += __shfl_sync(0xffffffffu, ic, 31);
        chb += __shfl_sync(0xffffffffu, in, 31);
      }
      return W;
    };
    const long long lo = W > 0 ? chunk_at_cost(range_lo(Ctot, a.num_ctas, cta)) : 0;
    const long long hi = W > 0 ? chunk_at_cost(range_lo(Ctot, a.num_ctas, cta + 1)) : 0;
    if (lane == 0) {
      *total_tiles = W;
      *total_cost = Ctot;
      *cost_chunk = cu_chunk;
    }
    // (blocks, length, q row) of request r, for every lane.
    auto req_info = [&](int r, int* len, int* row) -> int {
      int nbv = 0, lv = 0, rv = 0;
      if (r < 32 * kReqCache) {
        const int k = r >> 5;
#pragma unroll
        for (int m = 0; m < kReqCache; ++m)
          if (m == k) {
            nbv = c_nb[m];
            lv = c_len[m];
            rv = c_row[m];
          }
        nbv = __shfl_sync(0xffffffffu, nbv, r & 31);
        lv = __shfl_sync(0xffffffffu, lv, r & 31);
        rv = __shfl_sync(0xffffffffu, rv, r & 31);
      } else if (r < a.num_seqs) {
        nbv = request_blocks(a, r, &lv, &rv);
      }
      *len = lv;
      *row = rv;
      return nbv;
    };
    const uint64_t policy = l2_policy_evict_first();
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    int seg = 0, chunk = 0;
    bool ok = true;
    // Waits (lane 0) for a barrier phase; every lane learns the outcome.
    auto lane0_wait = [&](uint32_t b, uint32_t parity, int where) -> bool {
      int good = 1;
      if (lane == 0) {
        if (*fail_flag) good = 0;
        else if (!mbar_wait(b, parity)) { give_up(where); good = 0; }
      }
      return __shfl_sync(0xffffffffu, good, 0) != 0;
    };
    // Block ids of tiles 0 .. 63 of a request (lane L: tiles L and 32 + L).
    auto load_head = [&](int r, int nb, int& h0, int& h1) {
      const int32_t* rp = a.block_tables + static_cast<size_t>(r) * a.max_blocks_per_seq;
      h0 = (r < a.num_seqs && lane < nb) ? __ldg(rp + (lane >> a.tile_shift)) : 0;
      h1 = (r < a.num_seqs && 32 + lane < nb) ? __ldg(rp + ((32 + lane) >> a.tile_shift)) : 0;
    };
    if (lo < hi) {
      // Request holding chunk `lo`: scan the per-request chunk counts (and
      // split costs) 32 at a time.
      long long base = 0, cbase = 0;  // chunks and cost before request r0
      int r0 = -1;
      for (int rc = 0; rc < a.num_seqs && r0 < 0; rc += 32) {
        const int r = rc + lane;
        const int nc = (req_nb(r) + C::CB - 1) / C::CB;
        const long long nt = static_cast<long long>(nc) * a.num_kv_heads;
        const long long ct = nc > 0 ? a.num_kv_heads * (static_cast<long long>(cu_chunk) * nc + cu_seg) : 0;
        long long incl = nt, icl = ct;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long v = __shfl_up_sync(0xffffffffu, incl, o);
          const long long vc = __shfl_up_sync(0xffffffffu, icl, o);
          if (lane >= o) {
            incl += v;
            icl += vc;
          }
        }
        const unsigned hit = __ballot_sync(0xffffffffu, r < a.num_seqs && base + incl > lo);
        if (hit) {
          const int first = __ffs(hit) - 1;
          base += __shfl_sync(0xffffffffu, incl - nt, first);
          cbase += __shfl_sync(0xffffffffu, icl - ct, first);
          r0 = rc + first;
        } else {
          base += __shfl_sync(0xffffffffu, incl, 31);
          cbase += __shfl_sync(0xffffffffu, icl, 31);
        }
      }
      int r = r0, len = 0, row = 0;
      int nb = req_info(r, &len, &row);   // tiles of the request
      int nc = (nb + C::CB - 1) / C::CB;  // chunks of each of its pairs
      const long long off0 = lo - base;
      int kvh = static_cast<int>(off0 / nc);
      int cc = static_cast<int>(off0 % nc);  // first chunk of the range in the pair
      int b = cc * C::CB;
      long long t = lo;
      // Ids of the current request's blocks 0 .. 63 and of the next request's.
      int head0, head1, nhead0, nhead1;
      load_head(r, nb, head0, head1);
      int nlen = 0, nrow = 0;
      int nnb = req_info(r + 1, &nlen, &nrow);
      load_head(r + 1, nnb, nhead0, nhead1);
      while (t < hi && ok) {
        const int seg_c = static_cast<int>(min(hi - t, static_cast<long long>(nc - cc)));  // chunks
        const int seg_n = min(seg_c * C::CB, nb - b);                                       // tiles
        const int kind = (cc == 0 && seg_c == nc) ? kWhole : (cc > 0 ? kHead : kTail);
        const int slot = seg % C::SLOTS;
        // ---- segment record and q (slot reused once its epilogue is done)
        if (seg >= C::SLOTS && !lane0_wait(bar(B::SEGFREE + slot), ((seg / C::SLOTS) - 1) & 1, 20)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          TcSeg si;
          si.row = row;
          si.seq_len = len;
          si.npair = nc;
          si.b0 = b;
          si.nseg = seg_n;
          si.kind = kind;
          si.r = r;
          si.kvh = kvh;
          si.t0 = base + static_cast<long long>(kvh) * nc;
          si.c0 = cbase + static_cast<long long>(kvh) * (static_cast<long long>(cu_chunk) * nc + cu_seg) +
                  cu_seg;
          segs[slot] = si;
          mbar_arrive_expect_tx(bar(B::QFULL + slot), a.group * D * 2);
#pragma unroll
          for (int h = 0; h < C::HALVES; ++h)
            tma_load_3d(q_s + slot * C::QSLOT + h * (C::N * 128), &qmap, bar(B::QFULL + slot), 64 * h,
                        kvh * a.group, row, policy);
          *n_segs_issued = seg + 1;
        }
        // ---- block ids of tiles [win_b, win_b + 64) of the request
        const int32_t* rowp = a.block_tables + static_cast<size_t>(r) * a.max_blocks_per_seq;
        const int seg_end = b + seg_n;
        int cur32 = head0, nxt32 = head1, win_b = 0;
        if (b > 0) {  // only the first segment of a range can start mid-request
          win_b = b;
          cur32 = b + lane < seg_end ? __ldg(rowp + ((b + lane) >> a.tile_shift)) : 0;
          nxt32 = b + 32 + lane < seg_end ? __ldg(rowp + ((b + 32 + lane) >> a.tile_shift)) : 0;
        }
        // ---- chunks of 8 blocks: lane L < 8 copies the K of block L.
        const int nch = (seg_n + C::CB - 1) / C::CB;
        for (int c = 0; c < nch && ok; ++c) {
          int off = b + C::CB * c - win_b;  // 0, 8, 16 or 24
          if (off >= 32) {
            cur32 = nxt32;
            win_b += 32;
            off -= 32;
            const int gi = win_b + 32 + lane;
            nxt32 = gi < seg_end ? __ldg(rowp + (gi >> a.tile_shift)) : 0;
          }
          const int nbc = min(C::CB, seg_n - C::CB * c);
          const int vphys = __shfl_sync(0xffffffffu, cur32, (off + lane) & 31);
          const int kphys = vphys;
          // An id outside the pool is reported and read as wholly out of
          // bounds (TMA fills zeros).
          const bool kbad = static_cast<unsigned>(kphys) >= static_cast<unsigned>(a.num_blocks);
          const bool vbad = static_cast<unsigned>(vphys) >= static_cast<unsigned>(a.num_blocks);
          const int tile = b + C::CB * c + lane;  // this lane's tile
          const int krow = kbad ? a.num_blocks * a.block_size : tile_row(a, kphys, tile);
          const int vrow = vbad ? a.num_blocks * a.block_size : tile_row(a, vphys, tile);
          if (lane < nbc && vbad) record_error(a.status, PA_DEV_BAD_BLOCK_ID, r, vphys);
          const int st = chunk % C::NST;
          // K: refill once the S MMA of chunk - NST is done (that MMA also
          // follows P.V(chunk - 2 NST), so the V producer is done with the
          // chunk record this one replaces).
          if (chunk >= C::NST && !lane0_wait(bar(B::KFREE + st), ((chunk / C::NST) - 1) & 1, 21)) {
            ok = false;
            break;
          }
          int* rec = recs + (chunk % C::NREC) * 12;
          if (lane < C::CB) rec[lane] = vrow;
          if (lane == 0) {
            rec[8] = kvh;
            rec[9] = nbc;
            rec[10] = min(nbc * kBlockSize, len - (b + C::CB * c) * kBlockSize);  // valid tokens
            rec[11] = c == 0 ? slot + 1 : 0;  // first chunk of the segment in q slot `slot`
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar(B::CREC + chunk % C::NREC));
            mbar_arrive_expect_tx(bar(B::KFULL + st), nbc * (KV8 ? C::BLK8 : C::BLK));
          }
          __syncwarp();
          if (lane < nbc) {
            if constexpr (KV8)  // e4m3: 16 token rows of head_dim bytes, swizzled
              tma_load_3d(k_s + st * C::RSTAGE + lane * C::BLK8, &kmap, bar(B::KFULL + st), 0, kvh, krow,
                          policy);
            else
              tma_load_5d(k_s + st * C::STAGE + lane * C::BLK, &kmap, bar(B::KFULL + st), 0, 0, 0,
                          krow / 8, kvh, policy);
          }
          ++chunk;
          if (lane == 0) *n_chunks_issued = chunk;
        }
        t += seg_c;
        cc += seg_c;
        b = cc * C::CB;
        ++seg;
        if (cc == nc && t < hi) {  // next (request, kv head) pair
          cc = 0;
          b = 0;
          if (++kvh == a.num_kv_heads) {
            kvh = 0;
            base += static_cast<long long>(nc) * a.num_kv_heads;
            cbase += a.num_kv_heads * (static_cast<long long>(cu_chunk) * nc + cu_seg);
            ++r;
            if (nnb > 0) {  // the prefetched next request
              nb = nnb;
              len = nlen;
              row = nrow;
              head0 = nhead0;
              head1 = nhead1;
            } else {  // skip requests without decode blocks
              nb = 0;
              while (nb == 0 && r < a.num_seqs) {
                nb = req_info(r, &len, &row);
                if (nb == 0) ++r;
              }
              if (nb > 0) load_head(r, nb, head0, head1);
            }
            nc = (nb + C::CB - 1) / C::CB;
            if (nb == 0) {
              ok = false;  // cannot happen while t < hi
            } else {
              nnb = req_info(r + 1, &nlen, &nrow);
              load_head(r + 1, nnb, nhead0, nhead1);
            }
          }
        }
      }
    }
    // End of the chunk records (blocks = 0) for the V producer.
    if (ok && chunk >= C::NST &&
        !lane0_wait(bar(B::KFREE + chunk % C::NST), ((chunk / C::NST) - 1) & 1, 25))
      ok = false;
    if (ok && lane == 0) {
      recs[(chunk % C::NREC) * 12 + 9] = 0;
      mbar_arrive(bar(B::CREC + chunk % C::NREC));
    }
    // End record (no q load: a plain arrive completes the phase).
    if (ok) {
      const int slot = seg % C::SLOTS;
      if (seg >= C::SLOTS && !lane0_wait(bar(B::SEGFREE + slot), ((seg / C::SLOTS) - 1) & 1, 23))
        ok = false;
      if (ok && lane == 0) {
        segs[slot].kind = kEndSeg;
        mbar_arrive(bar(B::QFULL + slot));
      }
    }
    if (!ok && lane == 0) *fail_flag = 1;
  } else if (warp == 10) {
    // ========================================================== V producer
    // Follows the K producer's chunk records: V of block L of a chunk by lane L.
    const uint64_t policy = l2_policy_evict_first();
    if (lane == 0) tma_prefetch_desc(&vmap);
    auto warp_wait = [&](uint32_t b, uint32_t parity, int where) -> bool {
      if (__shfl_sync(0xffffffffu, *fail_flag, 0)) return false;
      const bool good = __all_sync(0xffffffffu, mbar_wait(b, parity) ? 1 : 0) != 0;
      if (!good && lane == 0) give_up(where);
      return good;
    };
    bool ok = true;
    for (int i = 0; ok; ++i) {
      const int rs = i % C::NREC;
      if (!(ok = warp_wait(bar(B::CREC + rs), (i / C::NREC) & 1, 24))) break;
      const int* rec = recs + rs * 12;
      const int nbc = rec[9];
      if (nbc == 0) break;
      const int kvh = rec[8];
      const int vrow = lane < C::CB ? rec[lane] : 0;
      const int st = i % C::NST;
      // V: refill once the P.V MMA of chunk i - NST is done.
      if (i >= C::NST && !(ok = warp_wait(bar(B::VFREE + st), ((i / C::NST) - 1) & 1, 22))) break;
      if (lane == 0) mbar_arrive_expect_tx(bar(B::VFULL + st), nbc * (KV8 ? C::BLK8 : C::BLK));
      __syncwarp();
      if (lane < nbc) {
        if constexpr (KV8)
          tma_load_3d(v_s + st * C::RSTAGE + lane * C::BLK8, &vmap, bar(B::VFULL + st), 0, kvh, vrow,
                      policy);
        else
          tma_load_5d(v_s + st * C::STAGE + lane * C::BLK, &vmap, bar(B::VFULL + st), 0, 0, 0, vrow / 8,
                      kvh, policy);
      }
      if (lane == 0) *n_v_issued = i + 1;
    }
    if (!ok && lane == 0) *fail_flag = 1;
  } else if (warp == 1) {
    // ========================================================== MMA issuer
    if (lane == 0) {
      bool ok = true;
      int j = 0, seg = 0;
      // The P.V MMA of the previous chunk, issued after the next S MMA so the
      // softmax of chunk j overlaps P.V(j - 1).
      int pv_j = -1, pv_seg = 0;
      bool pv_first = false, pv_last = false;
      auto issue_pv = [&]() -> bool {
        const int pb = pv_j & 1;
        const int st = pv_j % C::NST;
        const int ob = pv_seg & 1;
        const int cv = KV8 ? pv_j % C::NCV : 0;
        if (*fail_flag) return false;
        if (!mbar_wait(bar(B::PFULL + pb), (pv_j >> 1) & 1)) { give_up(30); return false; }
        if (!(KV8 ? mbar_wait(bar(B::VCFULL + cv), (pv_j / C::NCV) & 1)
                  : mbar_wait(bar(B::VFULL + st), (pv_j / C::NST) & 1))) {
          give_up(31);
          return false;
        }
        if (pv_first && pv_seg >= 2 && !mbar_wait(bar(B::OFREE + ob), ((pv_seg - 2) >> 1) & 1)) {
          give_up(32);
          return false;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::CB; ++kk) {
          // A = V^T of block kk (MN-major: head_dim halves 1 KB apart, its two
          // 8-token groups GSTRIDE apart); B = P^T tokens 16 kk .. 16 kk + 15.
          // (e4m3: the f16 V the converter warps wrote in the same layout)
          const uint32_t va = KV8 ? vc_s + cv * C::STAGE + kk * C::BLK : v_s + st * C::STAGE + kk * C::BLK;
          umma_bf16(tmem + 32 + ob * 16, sdesc_sw128(va, 1024, C::GSTRIDE),
                    sdesc_sw128(p_s + pb * C::PBUF + (kk >> 2) * (C::N * 128) + (kk & 3) * 32, 16, 1024),
                    C::IDESC_O, (pv_first && kk == 0) ? 0u : 1u);
        }
        umma_commit(bar(B::PVDONE + pb));
        umma_commit(bar(KV8 ? B::VCFREE + cv : B::VFREE + st));
        if (pv_last) umma_commit(bar(B::OFULL + ob));
        *n_pv_issued = pv_j + 1;
        return true;
      };
      while (ok) {
        const int slot = seg % C::SLOTS;
        if (*fail_flag || !mbar_wait(bar(B::QFULL + slot), (seg / C::SLOTS) & 1)) {
          if (!*fail_flag) give_up(33);
          ok = false;
          break;
        }
        const TcSeg si = segs[slot];
        if (si.kind == kEndSeg) break;
        // e4m3: q of the segment converted to f16 by the converter warps.
        if (KV8 && !mbar_wait(bar(B::QCONV + slot), (seg / C::SLOTS) & 1)) {
          give_up(35);
          ok = false;
          break;
        }
        const int nch = (si.nseg + C::CB - 1) / C::CB;
        for (int c = 0; c < nch && ok; ++c, ++j) {
          const int st = j % C::NST;
          const int ck = KV8 ? j % C::NCK : 0;
          const int sb = j & 1;
          if (*fail_flag || !(KV8 ? mbar_wait(bar(B::KCFULL + ck), (j / C::NCK) & 1)
                                  : mbar_wait(bar(B::KFULL + st), (j / C::NST) & 1))) {
            ok = false;
            break;
          }
          if (j >= 2 && !mbar_wait(bar(B::SFREE + sb), ((j - 2) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // A = K (128 tokens x head_dim), B = q (16 rows x head_dim).  bf16:
            // K-major in shared memory (8-token groups GSTRIDE apart, head_dim
            // halves 1 KB apart); e4m3: converted to f16 in TMEM (token = lane).
            const uint32_t qb = q_s + slot * C::QSLOT + (kk >> 2) * (C::N * 128) + (kk & 3) * 32;
            if constexpr (KV8) {
              umma_tmem_a(tmem + sb * 16, tmem + C::KCOL + ck * (D / 2) + kk * 8, sdesc_sw128(qb, 16, 1024),
                          C::IDESC_S, kk > 0 ? 1u : 0u);
            } else {
              const uint32_t ka = k_s + st * C::STAGE + (kk >> 2) * 1024 + (kk & 3) * 32;
              umma_bf16(tmem + sb * 16, sdesc_sw128(ka, 16, C::GSTRIDE), sdesc_sw128(qb, 16, 1024),
                        C::IDESC_S, kk > 0 ? 1u : 0u);
            }
          }
          umma_commit(bar(B::SFULL + sb));
          umma_commit(bar(KV8 ? B::KCFREE + ck : B::KFREE + st));
          *n_s_issued = j + 1;
          if (pv_j >= 0 && !(ok = issue_pv())) break;
          pv_j = j;
          pv_seg = seg;
          pv_first = c == 0;
          pv_last = c == nch - 1;
        }
        if (!ok) {
          if (!*fail_flag) give_up(34);
          break;
        }
        ++seg;
      }
      if (ok && pv_j >= 0) ok = issue_pv();
      if (!ok) *fail_flag = 1;
    }
    __syncwarp();
  } else if (warp < 6) {
    // ============================================================ softmax
    // Warp w owns TMEM lanes 32 (w % 4) .. + 31: token tl of every chunk.
    const int q4 = warp & 3;
    const int tl = q4 * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const int G = a.group;
    const float sl2 = a.scale_log2;
    const int neg_key = f2key(-INFINITY);
    uint32_t red_phase = 0;
    // Barrier of the four softmax warps (bounded).
    auto red_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B::RED));
      const int done = mbar_wait(bar(B::RED), red_phase & 1) ? 1 : 0;
      ++red_phase;
      return __all_sync(0xffffffffu, done) != 0;
    };
    auto all_wait = [&](int k, uint32_t parity) -> bool {
      if (__shfl_sync(0xffffffffu, *fail_flag, 0)) return false;
      return __all_sync(0xffffffffu, mbar_wait(bar(k), parity) ? 1 : 0) != 0;
    };
    bool ok = true;
    int j = 0, seg = 0;
    while (ok) {
      const int slot = seg % C::SLOTS;
      if (!(ok = all_wait(B::QFULL + slot, (seg / C::SLOTS) & 1))) break;
      const TcSeg si = segs[slot];
      if (si.kind == kEndSeg) break;
      const int nch = (si.nseg + C::CB - 1) / C::CB;
      const int ob = seg & 1;
      float m_ref[GM], l_run[GM];
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        m_ref[h] = kNegBigTc;
        l_run[h] = 0.f;
      }
      for (int c = 0; c < nch; ++c, ++j) {
        const int sb = j & 1;
        const int st = j % C::NST;
        const int tok0 = (si.b0 + C::CB * c) * kBlockSize;
        const int nbc = min(C::CB, si.nseg - C::CB * c);
        const int ntok = min(nbc * kBlockSize, si.seq_len - tok0);  // >= 1
        const bool valid = tl < ntok;
        if (!(ok = all_wait(B::SFULL + sb, (j >> 1) & 1))) break;
        tc_fence_after();
        float s[C::N];
        tmem_ld16(lane_base + sb * 16, s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B::SFREE + sb));
        // Chunk maximum of every head: one redux per warp, then across warps.
        int* rk = red_key + (j & 1) * 4 * GM;
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          const int k = __reduce_max_sync(0xffffffffu, (valid && h < G) ? f2key(s[h]) : neg_key);
          if (lane == 0) rk[q4 * GM + h] = k;
        }
        if (!(ok = red_sync())) break;
        bool need = false;
        float m_new[GM];
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          m_new[h] = m_ref[h];
          const int k = max(max(rk[h], rk[GM + h]), max(rk[2 * GM + h], rk[3 * GM + h]));
          const float mc = key2f(k) * sl2;
          if (h < G && (c == 0 || mc > m_ref[h] + kSlackTc)) {
            m_new[h] = mc;
            need = true;
          }
        }
        if (need) {
          float alpha[GM];
#pragma unroll
          for (int h = 0; h < GM; ++h) {
            alpha[h] = c == 0 ? 0.f : fast_exp2(m_ref[h] - m_new[h]);
            l_run[h] *= alpha[h];
            m_ref[h] = m_new[h];
          }
          if (c > 0) {
            // O^T must hold P.V(j - 1) before its columns are rescaled.
            if (!(ok = all_wait(B::PVDONE + ((j - 1) & 1), ((j - 1) >> 1) & 1))) break;
            tc_fence_after();
            float o[C::N];
            tmem_ld16(lane_base + 32 + ob * 16, o);
#pragma unroll
            for (int h = 0; h < GM; ++h) o[h] *= alpha[h];
            tmem_st16(lane_base + 32 + ob * 16, o);
          }
        }
        // P buffer sb was read by P.V(j - 2).
        if (j >= 2 && !(ok = all_wait(B::PVDONE + sb, ((j - 2) >> 1) & 1))) break;
        // Weights, rounded to bf16 as the MMA reads them; P^T row h, column tl
        // of the 128-byte-swizzled K-major layout.
        const uint32_t prow = p_s + sb * C::PBUF + (tl >> 6) * (C::N * 128);
        const uint32_t pchunk = static_cast<uint32_t>((tl & 63) >> 3);
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          const float p = (valid && h < G) ? fast_exp2(fmaf(s[h], sl2, -m_ref[h])) : 0.f;
          uint16_t pbits;
          if constexpr (KV8) {  // f16 products for e4m3 caches
            const __half ph = __float2half_rn(p);
            l_run[h] += __half2float(ph);
            pbits = __half_as_ushort(ph);
          } else {
            const __nv_bfloat16 pb = __float2bfloat16_rn(p);
            l_run[h] += __bfloat162float(pb);
            pbits = __bfloat16_as_ushort(pb);
          }
          const uint32_t r8 = h & 7;
          st_shared_u16(prow + (h >> 3) * 1024 + r8 * 128 + ((pchunk ^ r8) << 4) + (tl & 7) * 2, pbits);
        }
        // V rows of tokens past the context (or of blocks not loaded) may
        // hold NaN, which a zero weight does not cancel inside the MMA (the
        // converter warps write those rows as zeros for e4m3 caches).
        if (!KV8 && ntok < C::CT) {
          if (!(ok = all_wait(B::VFULL + st, (j / C::NST) & 1))) break;
          if (!valid) {
            const uint32_t vrow =
                v_s + st * C::STAGE + (tl >> 4) * C::BLK + ((tl >> 3) & 1) * C::GSTRIDE + (tl & 7) * 128;
#pragma unroll
            for (int h = 0; h < C::HALVES; ++h)
#pragma unroll
              for (int q = 0; q < 8; ++q)
                st_shared_v4(vrow + h * 1024 + q * 16, make_uint4(0u, 0u, 0u, 0u));
          }
        }
        fence_proxy_async_smem();  // P^T and zeroed V rows are read by the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B::PFULL + sb));
      }
      if (!ok) break;
      // Publish m and this warp's part of l for the epilogue warps.
      float* ml = seg_ml + slot * 5 * GM;
#pragma unroll
      for (int h = 0; h < GM; ++h) {
        float x = l_run[h];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) {
          ml[(1 + q4) * GM + h] = x;
          if (q4 == 0) ml[h] = m_ref[h];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B::LREADY + slot));
      ++seg;
    }
    if (!ok && lane == 0 && !*fail_flag) give_up(40);
  } else if (warp < 10) {
    // =========================================================== epilogue
    // Warp w owns TMEM lanes 32 (w % 4) .. + 31: row tl (head_dim index) of O^T.
    const int q4 = warp & 3;
    const int tl = q4 * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const int G = a.group;
    uint32_t ered_phase = 0;
    auto ered_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B::ERED));
      const int done = mbar_wait(bar(B::ERED), ered_phase & 1) ? 1 : 0;
      ++ered_phase;
      return __all_sync(0xffffffffu, done) != 0;
    };
    auto all_wait = [&](int k, uint32_t parity) -> bool {
      if (__shfl_sync(0xffffffffu, *fail_flag, 0)) return false;
      return __all_sync(0xffffffffu, mbar_wait(bar(k), parity) ? 1 : 0) != 0;
    };
    bool ok = true;
    int seg = 0;
    while (ok) {
      const int slot = seg % C::SLOTS;
      const int ob = seg & 1;
      if (!(ok = all_wait(B::QFULL + slot, (seg / C::SLOTS) & 1))) break;
      const TcSeg si = segs[slot];
      if (si.kind == kEndSeg) break;
      if (!(ok = all_wait(B::LREADY + slot, (seg / C::SLOTS) & 1))) break;
      if (!(ok = all_wait(B::OFULL + ob, (seg >> 1) & 1))) break;
      tc_fence_after();
      float o[C::N];
      tmem_ld16(lane_base + 32 + ob * 16, o);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B::OFREE + ob));
      const float* ml = seg_ml + slot * 5 * GM;
      const int head0 = si.kvh * G;
      const int pslot = si.kind == kTail ? 1 : 0;
      if (tl < D) {
#pragma unroll
        for (int h = 0; h < GM; ++h) {
          if (h < G) {
            const float L = (ml[GM + h] + ml[2 * GM + h]) + (ml[3 * GM + h] + ml[4 * GM + h]);
            const float v = o[h] * a.v_scale / L;  // v_scale: the e4m3 cache's V scale, else 1
            if (si.kind == kWhole) {
              a.out[(static_cast<size_t>(si.row) * a.num_heads + head0 + h) * D + tl] = __float2bfloat16_rn(v);
            } else {
              const size_t rec = (static_cast<size_t>(cta) * 2 + pslot) * G + h;
              a.part_o[rec * D + tl] = v;
              if (tl == 0) *reinterpret_cast<float2*>(a.part_ml + rec * 2) = make_float2(ml[h], L);
            }
          }
        }
      }
      if (si.kind != kWhole) {
        // Publish the partial; the last of the pair's contributors merges them.
        __threadfence();
        if (!(ok = ered_sync())) break;
        // The CTAs whose ranges hold the pair's first and last chunks.
        const long long Ct = *total_cost;
        const int c0 = cta_of_tile(Ct, a.num_ctas, si.c0);
        const int c1 = cta_of_tile(Ct, a.num_ctas, si.c0 + static_cast<long long>(*cost_chunk) * (si.npair - 1));
        if (tl == 0)
          *last_flag = contribute(a.counters + static_cast<size_t>(si.r) * a.num_kv_heads + si.kvh,
                                  a.epoch, c1 - c0 + 1, a.status, si.r) ? 1 : 0;
        if (!(ok = ered_sync())) break;
        if (*last_flag) {
          __threadfence();
          for (int it = tl; it < G * D; it += 128) {
            const int h = it / D;
            const int d = it % D;
            float M = kNegBigTc;
            for (int cc = c0; cc <= c1; ++cc) {
              const size_t rec = (static_cast<size_t>(cc) * 2 + (cc == c0 ? 1 : 0)) * G + h;
              M = fmaxf(M, __ldcg(a.part_ml + rec * 2));
            }
            float L = 0.f, acc = 0.f;
            for (int cc = c0; cc <= c1; ++cc) {
              const size_t rec = (static_cast<size_t>(cc) * 2 + (cc == c0 ? 1 : 0)) * G + h;
              const float2 m_l = __ldcg(reinterpret_cast<const float2*>(a.part_ml + rec * 2));
              const float wt = m_l.y * fast_exp2(m_l.x - M);
              L += wt;
              acc = fmaf(wt, __ldcg(a.part_o + rec * D + d), acc);
            }
            a.out[(static_cast<size_t>(si.row) * a.num_heads + head0 + h) * D + d] =
                __float2bfloat16_rn(acc / L);
          }
          if (tl == 0)
            release_pair(a.counters + static_cast<size_t>(si.r) * a.num_kv_heads + si.kvh);
        }
      }
      if (!(ok = ered_sync())) break;  // the slot's m, l and last_flag are free again
      if (lane == 0) mbar_arrive(bar(B::SEGFREE + slot));
      ++seg;
    }
    if (!ok && lane == 0 && !*fail_flag) give_up(50);
  } else if constexpr (KV8) {
    // ===================================================== e4m3 converter
    // Warp w owns TMEM lanes 32 (w % 4) .. + 31: token tl of every chunk.
    // Per chunk: K row tl -> f16 into TMEM lane tl (the A operand of S^T =
    // K Q^T, head_dim pairs along the columns); V row tl -> f16 into the
    // swizzled [8-token group][head_dim half][8 tokens][128 B] layout the
    // P.V product reads (rows of tokens past the context written as zeros);
    // at a segment's first chunk, that segment's q -> f16 in place.
    const int q4 = warp & 3;
    const int tl = q4 * 32 + lane;
    const int ct = tl;  // converter thread 0 .. 127
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    auto all_wait = [&](int k, uint32_t parity, int where) -> bool {
      if (__shfl_sync(0xffffffffu, *fail_flag, 0)) return false;
      const bool good = __all_sync(0xffffffffu, mbar_wait(bar(k), parity) ? 1 : 0) != 0;
      if (!good && lane == 0) give_up(where);
      return good;
    };
    bool ok = true;
    int seg = 0;
    int prev_ntok = 0;  // valid tokens of chunk i - 1 (its V is converted after K of chunk i)
    // Chunk i's K is converted before chunk i - 1's V, so that an S MMA never
    // waits behind the P.V products that free the converted V buffers.
    for (int i = 0; ok; ++i) {
      const int rs = i % C::NREC;
      if (!(ok = all_wait(B::CREC + rs, (i / C::NREC) & 1, 90))) break;
      const int* rec = recs + rs * 12;
      const int nbc = rec[9];
      const int ntok = rec[10];
      const int first = rec[11];
      if (nbc > 0) {
        const int st = i % C::NST, ck = i % C::NCK;
        if (first) {
          const int slot = first - 1;
          if (!(ok = all_wait(B::QFULL + slot, (seg / C::SLOTS) & 1, 91))) break;
          for (int u = ct; u < C::QSLOT / 16; u += 128) {
            const uint32_t addr = q_s + slot * C::QSLOT + u * 16;
            const uint4 w = ld_shared_v4(addr);
            st_shared_v4(addr, make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y),
                                          bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w)));
          }
          fence_proxy_async_smem();  // read by the tensor core
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B::QCONV + slot));
          ++seg;
        }
        if (!(ok = all_wait(B::KFULL + st, (i / C::NST) & 1, 92))) break;
        if (i >= C::NCK && !(ok = all_wait(B::KCFREE + ck, ((i / C::NCK) - 1) & 1, 93))) break;
        const uint32_t krow = k_s + st * C::RSTAGE + (tl >> 4) * C::BLK8;
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          uint32_t kw[32];  // head_dim 64 h .. 64 h + 63 as 32 f16 pairs
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 w = ld_shared_v4(krow + e8_chunk<D>(tl & 15, 4 * h + c));
            kw[8 * c + 0] = e4m3x2_to_f16x2(w.x);
            kw[8 * c + 1] = e4m3x2_to_f16x2(w.x >> 16);
            kw[8 * c + 2] = e4m3x2_to_f16x2(w.y);
            kw[8 * c + 3] = e4m3x2_to_f16x2(w.y >> 16);
            kw[8 * c + 4] = e4m3x2_to_f16x2(w.z);
            kw[8 * c + 5] = e4m3x2_to_f16x2(w.z >> 16);
            kw[8 * c + 6] = e4m3x2_to_f16x2(w.w);
            kw[8 * c + 7] = e4m3x2_to_f16x2(w.w >> 16);
          }
          tmem_st32_async(lane_base + C::KCOL + ck * (D / 2) + 32 * h, kw);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B::KCFULL + ck));
          mbar_arrive(bar(B::KFREE + st));  // the landed K stage may be refilled
        }
      }
      if (i > 0) {
        // V of chunk i - 1.
        const int j = i - 1, st = j % C::NST, cv = j % C::NCV;
        if (!(ok = all_wait(B::VFULL + st, (j / C::NST) & 1, 94))) break;
        if (j >= C::NCV && !(ok = all_wait(B::VCFREE + cv, ((j / C::NCV) - 1) & 1, 95))) break;
        const uint32_t vrow = v_s + st * C::RSTAGE + (tl >> 4) * C::BLK8;
        const uint32_t vdst = vc_s + cv * C::STAGE + (tl >> 4) * C::BLK + ((tl >> 3) & 1) * C::GSTRIDE +
                              (tl & 7) * 128;
        const bool valid = tl < prev_ntok;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint4 w = make_uint4(0u, 0u, 0u, 0u);
          if (valid) w = ld_shared_v4(vrow + e8_chunk<D>(tl & 15, c));
          // dims 16 c .. 16 c + 15: 16-byte units 2 (c % 4) and + 1 of head_dim half c / 4
          const uint4 lo = make_uint4(e4m3x2_to_f16x2(w.x), e4m3x2_to_f16x2(w.x >> 16),
                                      e4m3x2_to_f16x2(w.y), e4m3x2_to_f16x2(w.y >> 16));
          const uint4 hi = make_uint4(e4m3x2_to_f16x2(w.z), e4m3x2_to_f16x2(w.z >> 16),
                                      e4m3x2_to_f16x2(w.w), e4m3x2_to_f16x2(w.w >> 16));
          const int u = 2 * (c & 3);
          st_shared_v4(vdst + (c >> 2) * 1024 + ((u ^ (tl & 7)) * 16), lo);
          st_shared_v4(vdst + (c >> 2) * 1024 + (((u + 1) ^ (tl & 7)) * 16), hi);
        }
        fence_proxy_async_smem();  // read by the tensor core
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(B::VCFULL + cv));
          mbar_arrive(bar(B::VFREE + st));  // the landed V stage may be refilled
        }
      }
      prev_ntok = ntok;
      if (nbc == 0) break;  // end of the chunk records
    }
    if (!ok && lane == 0 && !*fail_flag) give_up(96);
  }

  __syncthreads();
  if (*fail_flag && tid == 0) {
    // Let copies and MMAs still in flight finish before TMEM is released
    // and the CTA leaves (bounded).
    const int n = *n_chunks_issued, nv = *n_v_issued;
    for (int i = max(0, n - C::NST); i < n; ++i)
      (void)mbar_wait(bar(B::KFULL + i % C::NST), (i / C::NST) & 1);
    for (int i = max(0, nv - C::NST); i < nv; ++i)
      (void)mbar_wait(bar(B::VFULL + i % C::NST), (i / C::NST) & 1);
    const int ns = *n_s_issued, npv = *n_pv_issued;
    if (ns > 0) (void)mbar_wait(bar(B::SFULL + ((ns - 1) & 1)), ((ns - 1) >> 1) & 1);
    if (npv > 0) (void)mbar_wait(bar(B::PVDONE + ((npv - 1) & 1)), ((npv - 1) >> 1) & 1);
    const int nq = *n_segs_issued;
    for (int i = max(0, nq - C::SLOTS); i < nq; ++i)
      (void)mbar_wait(bar(B::QFULL + i % C::SLOTS), (i / C::SLOTS) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // Deferred dependency: the CTA completes only after the previous grid.
  if (a.defer_griddep && tid == 0) griddep_wait();
}

template <int D, int GM, bool KV8>
cudaError_t launch_decode_tc_impl(const DecodeArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, cudaStream_t stream) {
  using C = TcCfg<D, GM, KV8>;
  static bool attr_set[64] = {false};  // per device: set once
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    const cudaError_t err = cudaFuncSetAttribute(paged_decode_tc_kernel<D, GM, KV8>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  return launch_overlapped(paged_decode_tc_kernel<D, GM, KV8>, dim3(a.num_ctas), dim3(C::THREADS), C::SMEM,
                           stream, qmap, kmap, vmap, a);
}

template <int D, bool KV8>
cudaError_t launch_decode_tc_d(const DecodeArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, cudaStream_t stream) {
  if (a.group <= 4) return launch_decode_tc_impl<D, 4, KV8>(a, qmap, kmap, vmap, stream);
  if (a.group <= 8) return launch_decode_tc_impl<D, 8, KV8>(a, qmap, kmap, vmap, stream);
  if (a.group <= 16) return launch_decode_tc_impl<D, 16, KV8>(a, qmap, kmap, vmap, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, int head_dim, bool kv8, cudaStream_t stream) {
  if (head_dim == 128)
    return kv8 ? launch_decode_tc_d<128, true>(a, qmap, kmap, vmap, stream)
               : launch_decode_tc_d<128, false>(a, qmap, kmap, vmap, stream);
  if (head_dim == 64)
    return kv8 ? launch_decode_tc_d<64, true>(a, qmap, kmap, vmap, stream)
               : launch_decode_tc_d<64, false>(a, qmap, kmap, vmap, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
