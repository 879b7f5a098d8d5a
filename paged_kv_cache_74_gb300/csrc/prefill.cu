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
// GB300 design.  One CTA of four warps owns 128 query rows of one q head of
// one request.  TMA with 128-byte swizzle loads the Q tile once and K/V
// tiles of 128 keys (eight 16-token blocks gathered through the block
// table) into a two-stage ring.  One thread issues the MMAs:
//   S = Q K^T   M = N = 128, K = head_dim, both operands K-major, into TMEM;
//   O_j = P V   M = 128, N = head_dim, K = 128 keys, P K-major from shared
//               memory, V MN-major exactly as TMA stored it.
// Each warp reads its 32 rows of S from TMEM (tcgen05.ld), applies the
// causal and length masks, updates (m, l), and writes P as bf16 into the
// swizzled layout the next MMA reads; the output accumulator stays in
// registers (O = alpha O + O_j per tile).  V rows of keys that are out of
// context or not loaded are zeroed first: they may hold NaN, and a zero
// weight does not cancel a NaN inside the MMA.
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr float kNegBigP = -1e30f;

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
  static constexpr int OFF_P = OFF_V + 2 * HALVES * CHUNK;     // 2 key halves
  static constexpr int OFF_BAR = OFF_P + 2 * CHUNK;            // q, kv[2], s, o
  static constexpr int OFF_MISC = OFF_BAR + 8 * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;            // + 1024-byte alignment slack
  static constexpr int THREADS = 128;
  static constexpr uint32_t TMEM_COLS = 256;                   // S at column 0, O_j at 128
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0);
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 1);
  static constexpr uint32_t KV_BLOCK_BYTES = 2 * HALVES * 16 * 128;  // K and V of one block
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <int D>
__global__ void __launch_bounds__(128, 1)
prefill_tile_kernel(const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  using C = PrefillCfg<D>;
  const int qt = blockIdx.x;
  const int head = blockIdx.y;
  const int r = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int q0 = a.query_start_loc[r];
  const int q_len = a.query_start_loc[r + 1] - q0;
  if (q_len <= 1 || qt * C::BM >= q_len) return;  // decode rows and empty tiles
  const int seq_len = a.seq_lens[r];
  if (q_len > seq_len || seq_len > a.max_seq_len || seq_len > a.max_blocks_per_seq * kBlockSize ||
      q_len > a.max_query_len || q0 < 0 || q0 + q_len > a.total_q) {
    if (tid == 0 && qt == 0 && head == 0)
      record_error(a.status, q_len > seq_len || q_len > a.max_query_len || q0 < 0 ||
                                     q0 + q_len > a.total_q
                                 ? PA_DEV_BAD_QUERY_LEN
                                 : PA_DEV_BAD_SEQ_LEN,
                   r, q_len > seq_len ? q_len : seq_len);
    return;
  }
  const int ctx = seq_len - q_len;
  const int row0 = qt * C::BM;                     // first query (within the request)
  const int rows = min(C::BM, q_len - row0);       // valid query rows of this tile
  const int kv_end = ctx + row0 + rows;            // keys [0, kv_end) are needed
  const int n_tiles = (kv_end + C::BN - 1) / C::BN;
  const int nblk_need = (kv_end + kBlockSize - 1) / kBlockSize;
  const int kvh = head / a.group;
  const int32_t* bt = a.block_tables + static_cast<size_t>(r) * a.max_blocks_per_seq;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // swizzle atoms
  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_s = sbase + C::OFF_Q;
  const uint32_t k_s = sbase + C::OFF_K;
  const uint32_t v_s = sbase + C::OFF_V;
  const uint32_t p_s = sbase + C::OFF_P;
  const uint32_t q_bar = sbase + C::OFF_BAR;
  const uint32_t kv_bar0 = q_bar + 8;
  const uint32_t s_bar = q_bar + 24;
  const uint32_t o_bar = q_bar + 32;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_MISC);

  if (tid == 0) {
    mbar_init(q_bar, 1);
    mbar_init(kv_bar0, 1);
    mbar_init(kv_bar0 + 8, 1);
    mbar_init(s_bar, 1);
    mbar_init(o_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_slot)), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const uint64_t policy = l2_policy_evict_first();

  // Block ids of K/V tile t: warp 0 lanes 0..7 each hold one.
  auto load_ids = [&](int t) -> int {
    const int b = t * 8 + lane;
    return (lane < 8 && t < n_tiles && b < nblk_need) ? __ldg(bt + b) : -1;
  };
  // Issue (thread 0) the TMA loads of K/V tile t into stage t % 2; `ids`
  // holds lane b's block id (warp 0 must be converged: shuffles inside).
  auto issue_kv = [&](int t, int ids) {
    int phys[8];
#pragma unroll
    for (int b = 0; b < 8; ++b) phys[b] = __shfl_sync(0xffffffffu, ids, b);
    if (lane == 0 && t < n_tiles) {
      const int st = t & 1;
      const int nb = min(8, nblk_need - t * 8);
      const uint32_t bar = kv_bar0 + 8 * st;
      mbar_arrive_expect_tx(bar, nb * C::KV_BLOCK_BYTES);
      for (int b = 0; b < nb; ++b) {
        int row_c = phys[b] * kBlockSize;
        if (static_cast<unsigned>(phys[b]) >= static_cast<unsigned>(a.num_blocks)) {
          record_error(a.status, PA_DEV_BAD_BLOCK_ID, r, phys[b]);
          row_c = a.num_blocks * kBlockSize;  // wholly out of bounds: TMA fills zeros
        }
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          tma_load_3d(k_s + (st * C::HALVES + h) * C::CHUNK + b * 2048, &kmap, bar, 64 * h, kvh,
                      row_c, policy);
          tma_load_3d(v_s + (st * C::HALVES + h) * C::CHUNK + b * 2048, &vmap, bar, 64 * h, kvh,
                      row_c, policy);
        }
      }
    }
  };

  int ids_next = 0;
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      mbar_arrive_expect_tx(q_bar, C::HALVES * C::CHUNK);
#pragma unroll
      for (int h = 0; h < C::HALVES; ++h)
        tma_load_3d(q_s + h * C::CHUNK, &qmap, q_bar, 64 * h, head, q0 + row0, policy);
    }
    issue_kv(0, load_ids(0));
    issue_kv(1, load_ids(1));
    ids_next = load_ids(2);
  }

  // Per-row online-softmax state; thread tid owns query row tid of the tile.
  const int i_row = tid;
  const int limit = min(ctx + row0 + i_row, kv_end - 1);  // last key this row may see
  const float sl2 = a.scale_log2;
  float m_run = kNegBigP, l_run = 0.f;
  float o_acc[D];
#pragma unroll
  for (int d = 0; d < D; ++d) o_acc[d] = 0.f;
  bool failed = false;

  for (int j = 0; j < n_tiles; ++j) {
    const int st = j & 1;
    // ---- S = Q K^T
    if (tid == 0) {
      bool ok = (j > 0 || mbar_wait(q_bar, 0)) && mbar_wait(kv_bar0 + 8 * st, (j >> 1) & 1);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks / 4) * C::CHUNK + (ks % 4) * 32;
          umma_bf16(tmem, sdesc_sw128(q_s + off, 16, 1024),
                    sdesc_sw128(k_s + st * C::HALVES * C::CHUNK + off, 16, 1024), C::IDESC_S,
                    ks > 0);
        }
        umma_commit(s_bar);
      } else {
        record_error(a.status, PA_DEV_WAIT_TIMEOUT, r, 10);
      }
    }
    const bool s_ok = mbar_wait(s_bar, j & 1);
    if (__syncthreads_or(!s_ok)) {
      failed = true;
      break;
    }
    tc_fence_after();

    // ---- masks, online softmax, P (bf16) into shared memory
    const int key0 = j * C::BN;
    const bool full_tile = key0 + C::BN - 1 <= ctx + row0 && key0 + C::BN <= seq_len;
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < C::BN / 32; ++c) {
      float sv[32];
      tmem_ld32(tmem_lane + c * 32, sv);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const bool ok = full_tile || key0 + c * 32 + e <= limit;
        mx = fmaxf(mx, ok ? sv[e] : -INFINITY);
      }
    }
    const float m_new = fmaxf(m_run, mx * sl2);
    const float alpha = fast_exp2(m_run - m_new);
    l_run *= alpha;
    m_run = m_new;
    float psum = 0.f;
#pragma unroll
    for (int c = 0; c < C::BN / 32; ++c) {
      float sv[32];
      tmem_ld32(tmem_lane + c * 32, sv);
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const bool ok0 = full_tile || key0 + c * 32 + e <= limit;
        const bool ok1 = full_tile || key0 + c * 32 + e + 1 <= limit;
        const float p0 = ok0 ? fast_exp2(fmaf(sv[e], sl2, -m_new)) : 0.f;
        const float p1 = ok1 ? fast_exp2(fmaf(sv[e + 1], sl2, -m_new)) : 0.f;
        pk[e / 2] = pack_bf16x2(p0, p1);
        psum += bf16_lo(pk[e / 2]) + bf16_hi(pk[e / 2]);  // the sum uses the rounded weights
      }
      // keys c*32 .. c*32+31 = 4 chunks of 8 in key half c / 2
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int chunk = (c % 2) * 4 + q;  // chunk within the 64-key half
        const uint32_t addr = p_s + (c / 2) * C::CHUNK + i_row * 128 + ((chunk ^ (i_row & 7)) * 16);
        st_shared_v4(addr, make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]));
      }
    }
    l_run += psum;
    // V rows of keys past the context or never loaded may hold NaN: zero them.
    const int kz = min(seq_len, kv_end) - key0;  // keys [kz, BN) of this tile are unused
    if (kz < C::BN) {
      const int nz = (C::BN - max(kz, 0)) * C::HALVES * 8;
      for (int idx = tid; idx < nz; idx += C::THREADS) {
        const int row = max(kz, 0) + idx / (C::HALVES * 8);
        const int h = (idx / 8) % C::HALVES;
        st_shared_v4(v_s + (st * C::HALVES + h) * C::CHUNK + row * 128 + (idx % 8) * 16,
                     make_uint4(0u, 0u, 0u, 0u));
      }
    }
    fence_proxy_async_smem();  // P and the zeroed rows are read by the tensor core
    tc_fence_before();
    __syncthreads();

    // ---- O_j = P V
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < C::BN / 16; ++ks) {
        umma_bf16(tmem + C::BN,
                  sdesc_sw128(p_s + (ks / 4) * C::CHUNK + (ks % 4) * 32, 16, 1024),
                  sdesc_sw128(v_s + st * C::HALVES * C::CHUNK + ks * 2048, C::CHUNK, 1024),
                  C::IDESC_O, ks > 0);
      }
      umma_commit(o_bar);
    }
    const bool o_ok = mbar_wait(o_bar, j & 1);
    if (__syncthreads_or(!o_ok)) {
      failed = true;
      break;
    }
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float ov[32];
      tmem_ld32(tmem_lane + C::BN + c * 32, ov);
#pragma unroll
      for (int e = 0; e < 32; ++e) o_acc[c * 32 + e] = fmaf(o_acc[c * 32 + e], alpha, ov[e]);
    }
    // Stage st is free (its MMAs are done): refill it with tile j + 2.
    if (warp == 0) {
      issue_kv(j + 2, ids_next);
      ids_next = load_ids(j + 3);
    }
    tc_fence_before();
    __syncthreads();  // S and O_j in TMEM may be overwritten now
  }

  if (!failed && i_row < rows) {
    const float inv = 1.f / l_run;
    __nv_bfloat16* dst = a.out + (static_cast<size_t>(q0 + row0 + i_row) * a.num_heads + head) * D;
#pragma unroll
    for (int d = 0; d < D; d += 8) {
      const uint4 v = make_uint4(pack_bf16x2(o_acc[d] * inv, o_acc[d + 1] * inv),
                                 pack_bf16x2(o_acc[d + 2] * inv, o_acc[d + 3] * inv),
                                 pack_bf16x2(o_acc[d + 4] * inv, o_acc[d + 5] * inv),
                                 pack_bf16x2(o_acc[d + 6] * inv, o_acc[d + 7] * inv));
      *reinterpret_cast<uint4*>(dst + d) = v;
    }
  }
  if (failed && tid == 0) {
    record_error(a.status, PA_DEV_WAIT_TIMEOUT, r, 11);
    // Let issued copies and MMAs finish before the CTA leaves (bounded).
    (void)mbar_wait(kv_bar0, 0);
    (void)mbar_wait(kv_bar0 + 8, 0);
    (void)mbar_wait(s_bar, 0);
    (void)mbar_wait(o_bar, 0);
  }
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
  const dim3 grid((a.max_query_len + C::BM - 1) / C::BM, a.num_heads, a.num_seqs);
  prefill_tile_kernel<D><<<grid, C::THREADS, C::SMEM, stream>>>(qmap, kmap, vmap, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int head_dim, cudaStream_t stream) {
  if (head_dim == 128) return launch_prefill_impl<128>(a, qmap, kmap, vmap, stream);
  if (head_dim == 64) return launch_prefill_impl<64>(a, qmap, kmap, vmap, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
