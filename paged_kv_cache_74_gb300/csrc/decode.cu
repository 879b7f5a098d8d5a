// decode.cu -- paged decode attention for sm_103a.
//
// Method ("vLLM 深度解析（二）：PagedAttention 核心机制"):
//   section 3.1  a request's token t lives in physical block
//                block_table[r][t / 16] at offset t % 16;
//   section 2.2  online softmax: a running (m, l, A) per query row, merged
//                tile by tile, O = A / l at the end;
//   section 3.2  masked scores of tokens >= seq_len are excluded and the V
//                of out-of-context slots is zeroed before it is used;
//   sections 3.2.7, 3.2.9, 3.3  long contexts are cut into partitions whose
//                (m_j, l_j, O_j) are merged by a second pass.
//
// GB300 design.  Decode is HBM-bound (about 2 FMAs per byte of KV at
// 4 q heads per kv head), so the K/V stream runs on CUDA cores, not tensor
// cores.  One CTA owns (partition, kv head, request) and serves every q head
// of that kv head, so each K/V byte is read from HBM once.  A producer warp
// reads the partition's block ids 32 at a time and issues one TMA tensor
// load per (block, kv head) tile of K and of V (16 tokens x head_dim, 4 KB at
// head_dim 128) into an 8-stage shared-memory ring guarded by mbarriers.
// Four consumer warps take every 4th block.  Inside a warp, T lanes share
// one token: each lane holds a 16-byte-chunk slice of head_dim for q (fp32,
// pre-scaled by scale * log2 e) and for its output accumulator, computes
// partial dot products for all q heads of the group, and a butterfly
// reduce-scatter leaves each lane with whole scores of a few (token, head)
// pairs; the exponentials are then computed once per score, not once per
// lane, and an all-gather hands the weights back for the P.V update.
// The running max is rescaled lazily: only when a new score exceeds the
// current reference by more than 2^8 (the final O = A / l is exact for any
// reference).  Partials are merged across the four warps in shared memory
// and either written as the final bf16 output (single partition) or as a
// normalised partial (m_j, l_j, O_j) for the merge kernel.
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr float kNegBig = -1e30f;      // finite stand-in for -inf in running maxima
constexpr float kRescaleSlack = 8.0f;  // log2 units

// Work split of one warp over one 16-token block (see the file comment).
template <int D, int GMAX>
struct DecodeCfg {
  static constexpr int T = (D == 128 && GMAX >= 4) ? 16 : 8;  // lanes per token
  static constexpr int NG = 32 / T;                            // token groups per warp
  static constexpr int NT = kBlockSize / NG;                   // tokens per group per block
  static constexpr int CPL = D / 8 / T;                        // 16-byte chunks per lane per row
  static constexpr int EL = CPL * 8;                           // head_dim elements per lane
  static constexpr int EP = EL / 2;                            // ... as float2 pairs
  static constexpr int SB = (NT * GMAX > 32) ? 32 / GMAX : NT; // tokens per sub-batch
  static constexpr int NSB = NT / SB;
  static constexpr int V = SB * GMAX;                          // partial scores per lane per sub-batch
  static constexpr int VPL = V >= T ? V / T : 1;               // whole scores per lane after the sum
  static constexpr int REP = V >= T ? 1 : T / V;               // lanes holding the same score
  static constexpr int LPH = T / GMAX;                         // lanes of a group per head
  static constexpr int CH = V / 4 > 0 ? V / 4 : 1;              // 16-byte chunks per transpose row
  static constexpr int NC = 4;                                 // consumer warps
  static constexpr int MINB = GMAX * EL > 32 ? 2 : 3;          // CTAs per SM the registers allow
  static constexpr int TILE = kBlockSize * D * 2;              // bytes of one (block, kv head) tile
  // The partial-score transpose (32 rows of V floats) reuses the warp's own
  // K tile once its q.k products are done, when it fits and no later
  // sub-batch still needs K; otherwise each warp gets a dedicated buffer.
  static constexpr bool XPOSE_IN_K = 32 * CH * 16 <= TILE && NSB == 1;
  static constexpr int XPOSE = XPOSE_IN_K ? 0 : 32 * CH * 16;
  static constexpr int STAGES = D == 128 ? 8 : 16;             // a multiple of NC (see below)
  static constexpr int SCRATCH = XPOSE + NG * V * 4;           // per warp: transpose + weights
  static constexpr int SCRATCH_AL = (SCRATCH + 127) / 128 * 128;
  static constexpr int COMB = NC * GMAX * (D + 2) * 4;         // cross-warp merge (aliases the ring)
  static constexpr int SMEM_RING = STAGES * 2 * TILE;
  static constexpr int SMEM_SCR = NC * SCRATCH_AL;
  static constexpr int SMEM = SMEM_RING + SMEM_SCR + 2 * STAGES * 8 + 16 + 1024;  // + align slack
  static constexpr int THREADS = (NC + 1) * 32;
  // Block i goes to stage i % STAGES and to warp i % NC.  With STAGES a
  // multiple of NC a stage is only ever used by one warp, so when a warp
  // waits on a stage the barrier is at most one phase behind and the
  // parity wait is unambiguous.
  static_assert(STAGES % NC == 0, "each ring stage must belong to one consumer warp");
  static_assert(COMB <= SMEM_RING, "merge buffer must fit in the ring");
  static_assert(SMEM <= 227 * 1024 && MINB * (SMEM + 1024) <= 228 * 1024,
                "shared memory must allow MINB CTAs per SM");
  static_assert(CPL >= 1 && GMAX <= T && NT % SB == 0 && V <= 32, "unsupported decode shape");
};

__device__ __forceinline__ float2 unpack2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <int D, int GMAX>
__global__ void __launch_bounds__(DecodeCfg<D, GMAX>::THREADS, DecodeCfg<D, GMAX>::MINB)
paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  using C = DecodeCfg<D, GMAX>;
  const int kvh = blockIdx.x;
  const int part = blockIdx.y;
  const int seq = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool reporter = threadIdx.x == 0 && part == 0 && kvh == 0;

  int row = seq;
  if (a.query_start_loc != nullptr) {
    const int q0 = a.query_start_loc[seq];
    const int q1 = a.query_start_loc[seq + 1];
    if (q1 - q0 != 1) return;  // not a decode row
    row = q0;
    if (row < 0 || row >= a.total_q) {
      if (reporter) record_error(a.status, PA_DEV_BAD_QUERY_LEN, seq, row);
      return;
    }
  }
  const int seq_len = a.seq_lens[seq];
  if (seq_len < 1 || seq_len > a.max_seq_len || seq_len > a.max_blocks_per_seq * kBlockSize) {
    if (reporter) record_error(a.status, PA_DEV_BAD_SEQ_LEN, seq, seq_len);
    return;
  }
  const int nblk_seq = (seq_len + kBlockSize - 1) / kBlockSize;
  const int b0 = part * a.partition_blocks;
  if (b0 >= nblk_seq) return;
  const int nblk = min(a.partition_blocks, nblk_seq - b0);
  const int nparts = (nblk_seq + a.partition_blocks - 1) / a.partition_blocks;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // TMA destinations want an aligned base: round up inside the (padded) allocation.
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* scratch = smem + C::SMEM_RING;
  uint64_t* bars = reinterpret_cast<uint64_t*>(scratch + C::SMEM_SCR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * C::STAGES);
  const uint32_t ring_s = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * C::STAGES;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == C::NC) {
    // ------------------------------------------------------------ producer
    const int32_t* bt = a.block_tables + static_cast<size_t>(seq) * a.max_blocks_per_seq + b0;
    const uint64_t policy = l2_policy_evict_first();
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    int my_id = 0;
    int issued = 0;
    for (int i = 0; i < nblk; ++i) {
      if ((i & 31) == 0) {
        const int j = i + lane;
        my_id = j < nblk ? __ldg(bt + j) : 0;
      }
      const int phys = __shfl_sync(0xffffffffu, my_id, i & 31);
      int stop = 0;
      if (lane == 0) {
        const int s = i % C::STAGES;
        if (i >= C::STAGES && !mbar_wait(empty0 + 8 * s, ((i / C::STAGES) - 1) & 1)) {
          record_error(a.status, PA_DEV_WAIT_TIMEOUT, seq, 1);
          *abort_flag = 1;
        }
        if (*abort_flag) {
          stop = 1;
        } else {
          int row0 = phys * kBlockSize;
          if (static_cast<unsigned>(phys) >= static_cast<unsigned>(a.num_blocks)) {
            record_error(a.status, PA_DEV_BAD_BLOCK_ID, seq, phys);
            row0 = a.num_blocks * kBlockSize;  // wholly out of bounds: TMA fills zeros
          }
          const uint32_t full = full0 + 8 * s;
          mbar_arrive_expect_tx(full, 2 * C::TILE);
          tma_load_3d(ring_s + (2 * s) * C::TILE, &kmap, full, 0, kvh, row0, policy);
          tma_load_3d(ring_s + (2 * s + 1) * C::TILE, &vmap, full, 0, kvh, row0, policy);
          issued = i + 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) break;
    }
    if (lane == 0 && *abort_flag) {
      // Let the copies already in flight land before the CTA can exit.
      for (int i = max(0, issued - C::STAGES); i < issued; ++i)
        (void)mbar_wait(full0 + 8 * (i % C::STAGES), (i / C::STAGES) & 1);
    }
    return;
  }

  // -------------------------------------------------------------- consumer
  const int g = lane / C::T;
  const int li = lane % C::T;
  const int head0 = kvh * a.group;
  uint8_t* my_scratch = scratch + warp * C::SCRATCH_AL;
  float* pbuf = reinterpret_cast<float*>(my_scratch + C::XPOSE);  // [NG][V] weights

  // q of every head of the group over this lane's slice of head_dim, as
  // float2 pairs, pre-scaled by scale * log2(e).
  float2 q2[GMAX][C::EP];
  {
    const __nv_bfloat16* qrow = a.q + (static_cast<size_t>(row) * a.num_heads + head0) * D;
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
#pragma unroll
      for (int j = 0; j < C::CPL; ++j) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (h < a.group) w = __ldg(reinterpret_cast<const uint4*>(qrow + h * D + (li + C::T * j) * 8));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack2(ws[e]);
          q2[h][j * 4 + e] = make_float2(f.x * a.scale_log2, f.y * a.scale_log2);
        }
      }
    }
  }

  float2 o2[GMAX][C::EP];
#pragma unroll
  for (int h = 0; h < GMAX; ++h)
#pragma unroll
    for (int e = 0; e < C::EP; ++e) o2[h][e] = make_float2(0.f, 0.f);
  float my_m = kNegBig;  // running max (log2 units) of this lane's head, same on all its lanes
  float my_l = 0.f;      // this lane's share of the running exp-sum
  const int idx0 = (li * C::V) / C::T;
  const int my_h = idx0 / C::SB;
  const int my_k0 = idx0 % C::SB;
  const bool head_real = my_h < a.group;
  const bool l_owner = (li % C::REP) == 0;

  for (int i = warp; i < nblk; i += C::NC) {
    const int s = i % C::STAGES;
    // Every branch below is taken by the whole warp.
    if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
    const int landed = mbar_wait(full0 + 8 * s, (i / C::STAGES) & 1) ? 1 : 0;
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) {
        record_error(a.status, PA_DEV_WAIT_TIMEOUT, seq, 2);
        *abort_flag = 1;
      }
      break;
    }
    const uint32_t kt = ring_s + (2 * s) * C::TILE;
    const uint32_t vt = kt + C::TILE;
    // Transpose rows: lane L's 16-byte chunk c sits at chunk c ^ (L % CH) of
    // row L (bank-conflict-free 16-byte stores from 8 consecutive lanes).
    float* xpose = C::XPOSE_IN_K ? reinterpret_cast<float*>(smem + (2 * s) * C::TILE)
                                 : reinterpret_cast<float*>(my_scratch);
    const int tok0 = (b0 + i) * kBlockSize;
    const bool tail = tok0 + kBlockSize > seq_len;

#pragma unroll
    for (int sb = 0; sb < C::NSB; ++sb) {
      // Partial q.k over this lane's head_dim slice, every head, SB tokens.
      float x[C::V];
#pragma unroll
      for (int kk = 0; kk < C::SB; ++kk) {
        const int t = (sb * C::SB + kk) * C::NG + g;
        uint4 kw[C::CPL];
#pragma unroll
        for (int j = 0; j < C::CPL; ++j) kw[j] = ld_shared_v4(kt + t * (D * 2) + (li + C::T * j) * 16);
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          float2 acc = make_float2(0.f, 0.f);
#pragma unroll
          for (int j = 0; j < C::CPL; ++j) {
            acc = __ffma2_rn(q2[h][j * 4 + 0], unpack2(kw[j].x), acc);
            acc = __ffma2_rn(q2[h][j * 4 + 1], unpack2(kw[j].y), acc);
            acc = __ffma2_rn(q2[h][j * 4 + 2], unpack2(kw[j].z), acc);
            acc = __ffma2_rn(q2[h][j * 4 + 3], unpack2(kw[j].w), acc);
          }
          x[h * C::SB + kk] = acc.x + acc.y;
        }
      }
      // Sum the partials of the T lanes of a group through shared memory:
      // lane L writes row L; each lane then adds up its VPL columns.
      __syncwarp();  // every lane is done reading K before the rows overwrite it
      if constexpr (C::V >= 4) {
#pragma unroll
        for (int c = 0; c < C::CH; ++c)
          *reinterpret_cast<float4*>(xpose + lane * (C::CH * 4) + ((c ^ (lane % C::CH)) * 4)) =
              make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
      } else {
#pragma unroll
        for (int v = 0; v < C::V; ++v) xpose[lane * 4 + v] = x[v];
      }
      __syncwarp();
      float sc[C::VPL];
#pragma unroll
      for (int u = 0; u < C::VPL; ++u) sc[u] = 0.f;
#pragma unroll
      for (int l2 = 0; l2 < C::T; ++l2) {
        const int r = g * C::T + l2;
        const float* src = C::V >= 4
            ? xpose + r * (C::CH * 4) + (((idx0 / 4) ^ (r % C::CH)) * 4) + (idx0 % 4)
            : xpose + r * 4 + idx0;
        if constexpr (C::VPL == 2) {
          const float2 v2 = *reinterpret_cast<const float2*>(src);
          sc[0] += v2.x;
          sc[1] += v2.y;
        } else {
#pragma unroll
          for (int u = 0; u < C::VPL; ++u) sc[u] += src[u];
        }
      }
      // Mask tokens past seq_len (and padding heads), then the lazy max.
      float smax = -INFINITY;
#pragma unroll
      for (int u = 0; u < C::VPL; ++u) {
        const int t = (sb * C::SB + my_k0 + u) * C::NG + g;
        const bool ok = head_real && (tok0 + t < seq_len);
        sc[u] = ok ? sc[u] : -INFINITY;
        smax = fmaxf(smax, sc[u]);
      }
      if (__any_sync(0xffffffffu, smax > my_m + kRescaleSlack)) {
        float bm = smax;
#pragma unroll
        for (int b = 1; b < C::LPH; b <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, b));
#pragma unroll
        for (int b = C::T; b < 32; b <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, b));
        const float m_new = fmaxf(my_m, bm);
        const float alpha = fast_exp2(my_m - m_new);
        my_l *= alpha;
        my_m = m_new;
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          const float ah = __shfl_sync(0xffffffffu, alpha, h * C::LPH);
          const float2 a2 = make_float2(ah, ah);
#pragma unroll
          for (int e = 0; e < C::EP; ++e) o2[h][e] = __fmul2_rn(o2[h][e], a2);
        }
      }
      float psum = 0.f;
#pragma unroll
      for (int u = 0; u < C::VPL; ++u) {
        sc[u] = fast_exp2(sc[u] - my_m);
        psum += sc[u];
      }
      my_l += l_owner ? psum : 0.f;
      // Hand the weights to every lane of the group.
#pragma unroll
      for (int u = 0; u < C::VPL; ++u) pbuf[g * C::V + idx0 + u] = sc[u];
      __syncwarp();
      float p[C::V];
#pragma unroll
      for (int v = 0; v < C::V; v += 4) {
        const float4 f = *reinterpret_cast<const float4*>(pbuf + g * C::V + v);
        p[v] = f.x; p[v + 1] = f.y; p[v + 2] = f.z; p[v + 3] = f.w;
      }
      // A += p v over this sub-batch's tokens.
#pragma unroll
      for (int kk = 0; kk < C::SB; ++kk) {
        const int t = (sb * C::SB + kk) * C::NG + g;
        uint4 vw[C::CPL];
#pragma unroll
        for (int j = 0; j < C::CPL; ++j) vw[j] = ld_shared_v4(vt + t * (D * 2) + (li + C::T * j) * 16);
        if (tail && tok0 + t >= seq_len) {
#pragma unroll
          for (int j = 0; j < C::CPL; ++j) vw[j] = make_uint4(0u, 0u, 0u, 0u);  // may hold NaN
        }
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          const float2 pp = make_float2(p[h * C::SB + kk], p[h * C::SB + kk]);
#pragma unroll
          for (int j = 0; j < C::CPL; ++j) {
            o2[h][j * 4 + 0] = __ffma2_rn(pp, unpack2(vw[j].x), o2[h][j * 4 + 0]);
            o2[h][j * 4 + 1] = __ffma2_rn(pp, unpack2(vw[j].y), o2[h][j * 4 + 1]);
            o2[h][j * 4 + 2] = __ffma2_rn(pp, unpack2(vw[j].z), o2[h][j * 4 + 2]);
            o2[h][j * 4 + 3] = __ffma2_rn(pp, unpack2(vw[j].w), o2[h][j * 4 + 3]);
          }
        }
      }
      __syncwarp();  // the next sub-batch rewrites the scratch rows
    }
    // The stage is refilled by TMA (async proxy) after this release; order
    // this warp's generic-proxy writes into it (the transpose) before that.
    if (C::XPOSE_IN_K) fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * s);
  }

  // ------------------------------------------------- merge inside the warp
  float lsum = my_l;
#pragma unroll
  for (int b = 1; b < C::LPH; b <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, b);
#pragma unroll
  for (int b = C::T; b < 32; b <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, b);
#pragma unroll
  for (int h = 0; h < GMAX; ++h)
#pragma unroll
    for (int e = 0; e < C::EP; ++e)
#pragma unroll
      for (int b = C::T; b < 32; b <<= 1) {
        o2[h][e].x += __shfl_xor_sync(0xffffffffu, o2[h][e].x, b);
        o2[h][e].y += __shfl_xor_sync(0xffffffffu, o2[h][e].y, b);
      }
  // The merge buffer aliases the ring: wait until every warp is done with
  // it.  Every block was issued and consumed unless the CTA aborted (then
  // copies may be in flight and nothing more is written).
  named_barrier_sync(1, C::NC * 32);
  if (*abort_flag) return;
  float* comb_o = reinterpret_cast<float*>(smem);          // [NC][GMAX][D]
  float* comb_ml = comb_o + C::NC * GMAX * D;               // [NC][GMAX][2]
  if (g == 0) {
#pragma unroll
    for (int h = 0; h < GMAX; ++h)
#pragma unroll
      for (int j = 0; j < C::CPL; ++j) {
        float4* dst = reinterpret_cast<float4*>(comb_o + (warp * GMAX + h) * D + (li + C::T * j) * 8);
        dst[0] = make_float4(o2[h][j * 4 + 0].x, o2[h][j * 4 + 0].y, o2[h][j * 4 + 1].x, o2[h][j * 4 + 1].y);
        dst[1] = make_float4(o2[h][j * 4 + 2].x, o2[h][j * 4 + 2].y, o2[h][j * 4 + 3].x, o2[h][j * 4 + 3].y);
      }
    if (li % C::LPH == 0) {
      comb_ml[(warp * GMAX + my_h) * 2 + 0] = my_m;
      comb_ml[(warp * GMAX + my_h) * 2 + 1] = lsum;
    }
  }
  named_barrier_sync(1, C::NC * 32);

  // ------------------------------------------------ merge across the warps
  for (int it = threadIdx.x; it < a.group * (D / 2); it += C::NC * 32) {
    const int h = it / (D / 2);
    const int d = (it % (D / 2)) * 2;
    float M = kNegBig;
#pragma unroll
    for (int w = 0; w < C::NC; ++w) M = fmaxf(M, comb_ml[(w * GMAX + h) * 2]);
    float L = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
    for (int w = 0; w < C::NC; ++w) {
      const float wt = fast_exp2(comb_ml[(w * GMAX + h) * 2] - M);
      L = fmaf(wt, comb_ml[(w * GMAX + h) * 2 + 1], L);
      const float2 ov = *reinterpret_cast<const float2*>(comb_o + (w * GMAX + h) * D + d);
      o0 = fmaf(wt, ov.x, o0);
      o1 = fmaf(wt, ov.y, o1);
    }
    const float inv = 1.f / L;
    const int head = head0 + h;
    if (nparts == 1) {
      *reinterpret_cast<__nv_bfloat162*>(a.out + (static_cast<size_t>(row) * a.num_heads + head) * D + d) =
          __floats2bfloat162_rn(o0 * inv, o1 * inv);
    } else {
      const size_t base = (static_cast<size_t>(seq) * a.num_heads + head) * a.max_parts + part;
      *reinterpret_cast<float2*>(a.part_o + base * D + d) = make_float2(o0 * inv, o1 * inv);
      if (d == 0) *reinterpret_cast<float2*>(a.part_ml + base * 2) = make_float2(M, L);
    }
  }
}

// Second pass for requests split into several partitions:
//   M = max_j m_j,  w_j = l_j 2^{m_j - M},  O = sum_j w_j O_j / sum_j w_j.
template <int D>
__global__ void __launch_bounds__(D) merge_partitions_kernel(const DecodeArgs a) {
  const int head = blockIdx.x;
  const int seq = blockIdx.y;
  const int d = threadIdx.x;
  int row = seq;
  if (a.query_start_loc != nullptr) {
    const int q0 = a.query_start_loc[seq];
    if (a.query_start_loc[seq + 1] - q0 != 1) return;
    row = q0;
    if (row < 0 || row >= a.total_q) return;
  }
  const int seq_len = a.seq_lens[seq];
  if (seq_len < 1 || seq_len > a.max_seq_len || seq_len > a.max_blocks_per_seq * kBlockSize) return;
  const int nblk_seq = (seq_len + kBlockSize - 1) / kBlockSize;
  const int nparts = (nblk_seq + a.partition_blocks - 1) / a.partition_blocks;
  if (nparts <= 1) return;
  const size_t base = (static_cast<size_t>(seq) * a.num_heads + head) * a.max_parts;
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml) + base;
  const float* po = a.part_o + base * D + d;
  float M = kNegBig;
  for (int p = 0; p < nparts; ++p) M = fmaxf(M, ml[p].x);
  float L = 0.f, acc = 0.f;
#pragma unroll 4
  for (int p = 0; p < nparts; ++p) {
    const float2 v = ml[p];
    const float w = v.y * fast_exp2(v.x - M);
    L += w;
    acc = fmaf(w, po[static_cast<size_t>(p) * D], acc);
  }
  a.out[(static_cast<size_t>(row) * a.num_heads + head) * D + d] = __float2bfloat16_rn(acc / L);
}

template <int D, int GMAX>
cudaError_t launch_decode_impl(const DecodeArgs& a, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, cudaStream_t stream) {
  using C = DecodeCfg<D, GMAX>;
  cudaError_t err = cudaFuncSetAttribute(paged_decode_kernel<D, GMAX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(paged_decode_kernel<D, GMAX>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
  if (err != cudaSuccess) return err;
  const dim3 grid(a.num_kv_heads, a.max_parts, a.num_seqs);
  paged_decode_kernel<D, GMAX><<<grid, C::THREADS, C::SMEM, stream>>>(kmap, vmap, a);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (a.max_parts > 1) {
    merge_partitions_kernel<D><<<dim3(a.num_heads, a.num_seqs), D, 0, stream>>>(a);
    err = cudaGetLastError();
  }
  return err;
}

}  // namespace

int decode_gmax(int group) {
  if (group <= 1) return 1;
  if (group <= 2) return 2;
  if (group <= 4) return 4;
  if (group <= 8) return 8;
  return 0;
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          int head_dim, cudaStream_t stream) {
  const int gmax = decode_gmax(a.group);
#define PA_DECODE_CASE(DD, GG) \
  if (head_dim == DD && gmax == GG) return launch_decode_impl<DD, GG>(a, kmap, vmap, stream);
  PA_DECODE_CASE(128, 1) PA_DECODE_CASE(128, 2) PA_DECODE_CASE(128, 4) PA_DECODE_CASE(128, 8)
  PA_DECODE_CASE(64, 1) PA_DECODE_CASE(64, 2) PA_DECODE_CASE(64, 4) PA_DECODE_CASE(64, 8)
#undef PA_DECODE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
