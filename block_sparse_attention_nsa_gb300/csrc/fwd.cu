// fwd.cu -- forward of NSA selected attention on sm_103a.
//
// Loop order follows "FSA: An Alternative Efficient Implementation of Native
// Sparse Attention Kernel" (key design 1): the outer loop is over (KV head, KV
// block) segments of the index, the inner one over 128-row tiles of the query
// rows (token, query head) that selected the block, so the MMA's M dimension is
// filled by gathered queries and no GQA-group padding is needed.
//
//   fwd_main  : per tile, S = Q K_b^T (tcgen05, TMEM accumulator, M = 128,
//               N = B_K), masked row max m and P = exp2(S*scale*log2e - m) in
//               registers, O = P V_b (tcgen05, N = d).  The unnormalised partial
//               O and its (m, l = fp32 sum of P) go to the compact buffer at the pair's
//               position (O_i of key design 2), so a tile's output is one
//               contiguous block of memory.
//   fwd_merge : per (token, query head), the <= T partials are combined with
//               log-sum-exp weights into out and lse.  Carrying (m, l) with each
//               partial replaces the separate statistics kernel of key design 4:
//               every partial is rescaled once, at merge time, by exp2(m - M).
#include "common.cuh"

namespace nsa {

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pipeline depths per (d, B_K), bounded by 227 KB of shared memory and 512 TMEM
// columns: Q stages (a Q stage also stages the tile's 16-bit output), K/V stages,
// P buffers, O accumulators (TMEM).
__host__ __device__ constexpr int fwd_qs(int d, int bk) {
  return d == 64 ? 4 : (d == 128 ? 3 : (bk == 128 ? 1 : 2));
}
__host__ __device__ constexpr int fwd_kvs(int d, int bk) {
  return (d == 64 || (d == 128 && bk <= 64)) ? 2 : 1;
}
__host__ __device__ constexpr int fwd_ps(int d, int bk) { return (d == 256 && bk == 128) ? 1 : 2; }
__host__ __device__ constexpr int fwd_os(int d) { return d == 256 ? 1 : 2; }

template <int D, int BK>
struct FwdSmem {
  static constexpr int QS = fwd_qs(D, BK), KVS = fwd_kvs(D, BK), PS = fwd_ps(D, BK),
                       OS = fwd_os(D);
  static constexpr int kPCols = BK < 64 ? 64 : BK;
  static constexpr uint32_t kQ = 128u * D * 2u;            // one Q stage (and output staging)
  static constexpr uint32_t kK = uint32_t(BK) * D * 2u;     // one K (or V) stage
  static constexpr uint32_t kP = 128u * kPCols * 2u;        // one P buffer
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + QS * kQ;
  static constexpr uint32_t kOffV = kOffK + KVS * kK;
  static constexpr uint32_t kOffP = kOffV + KVS * kK;
  static constexpr uint32_t kBytes = kOffP + PS * kP + 1024;   // + alignment slack
  static_assert(kBytes <= 227u * 1024u, "shared memory budget");
  static_assert(2 * BK + OS * D <= 512, "TMEM budget");
  static constexpr uint32_t kTmemCols = 512;
};

constexpr int kFwdThreads = 384;   // warp 0 MMA, warp 2 TMA producer, warps 4-11 two softmax WGs

// Persistent, warp-specialised forward main kernel (one CTA per SM).
//   warp 2 (lane 0 + lanes for row coordinates): TMA loads -- K_b and V_b tiles
//     (3-D tensor maps, once per segment) and the 128 gathered Q rows of each
//     tile (tile::gather4 of four rows at a time), 128-byte swizzled;
//   warp 0 (one thread): tcgen05 MMAs S(i) = Q K^T into TMEM slot i % 2 and
//     O(i) = P V into an O accumulator, issued as S(0), S(1), O(0), S(2), O(1), ...;
//   warps 4-7 / 8-11: softmax of even / odd tiles (row max, exp2, P in 16-bit
//     to shared memory, fp32 row sum) and their epilogue (O from TMEM to 16-bit,
//     staged in the tile's Q stage, one bulk store of the tile's contiguous
//     compact-buffer rows, (m, l) per row).
// mbarriers hand each buffer between roles; every wait is bounded.
template <int D, int BK, bool kFp16>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_main_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, Params p) {
  using L = FwdSmem<D, BK>;
  constexpr int QS = L::QS, KVS = L::KVS, PS = L::PS, OS = L::OS;
  constexpr int kCB = D / 64;                      // 64-column blocks per row
  constexpr uint32_t kIdescS = idesc_f16(128, BK, false, false, kFp16);
  constexpr uint32_t kIdescO = idesc_f16(128, D, false, true, kFp16);

  extern __shared__ uint8_t smem_raw[];
  // Barriers a softmax warpgroup waits on (s_full, p_empty, o_full) are per warpgroup
  // (index i & 1) whatever the buffer counts, so no waiter is ever two phases ahead.
  __shared__ uint64_t q_full[QS], q_empty[QS], kv_full[KVS], kv_empty[KVS], s_full[2],
      p_full[PS], p_empty[2], o_full[2], o_free[OS];
  __shared__ uint32_t tmem_base;
  __shared__ int fail;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sQ0 = smem_u32(smem + L::kOffQ), sK0 = smem_u32(smem + L::kOffK),
                 sV0 = smem_u32(smem + L::kOffV), sP0 = smem_u32(smem + L::kOffP);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 0) tmem_alloc(&tmem_base, L::kTmemCols);
  if (tid == 32) {
    for (int i = 0; i < QS; ++i) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1); }
    for (int i = 0; i < KVS; ++i) { mbar_init(&kv_full[i], 1); mbar_init(&kv_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_empty[i], 1);
      mbar_init(&o_full[i], 1);
    }
    for (int i = 0; i < PS; ++i) mbar_init(&p_full[i], 128);
    for (int i = 0; i < OS; ++i) mbar_init(&o_free[i], 128);
    fail = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS0 = tmem_base, tO0 = tmem_base + 2 * BK;

  const int nb = *p.nb;
  const int nseg = p.h_k * nb;
  const int total_tiles = p.tile_off[nseg];
  const int per_cta = (total_tiles + gridDim.x - 1) / gridDim.x;
  const int t_begin = min(total_tiles, static_cast<int>(blockIdx.x) * per_cta);
  const int n = min(total_tiles, t_begin + per_cta) - t_begin;

  if (warp == 2) {
    // ------------------------------ producer ------------------------------
    if (n > 0) {
      TileCursor cur;
      cur.start(p, nb, t_begin);
      const int oob_row = p.n * p.h_q;     // zero-filled by the tensor map
      for (int i = 0; i < n; ++i) {
        cur.set(p, t_begin + i);
        if (cur.new_seg) {
          const int ks = cur.jseg % KVS;
          if (cur.jseg >= KVS) mbar_wait_sticky(&kv_empty[ks], ((cur.jseg / KVS) - 1) & 1, p.status, &fail);
          if (lane == 0) {
            mbar_arrive_expect_tx(&kv_full[ks], 2u * L::kK);
#pragma unroll
            for (int cb = 0; cb < kCB; ++cb) {
              tma_load_3d(sK0 + ks * L::kK + cb * BK * 128, &tm_k, cb * 64, cur.h, cur.key0, &kv_full[ks]);
              tma_load_3d(sV0 + ks * L::kK + cb * BK * 128, &tm_v, cb * 64, cur.h, cur.key0, &kv_full[ks]);
            }
          }
        }
        const int qs = i % QS;
        if (i >= QS) mbar_wait_sticky(&q_empty[qs], ((i / QS) - 1) & 1, p.status, &fail);
        if (lane == 0) mbar_arrive_expect_tx(&q_full[qs], L::kQ);
        __syncwarp();
        int rows[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = lane * 4 + j;
          if (r < cur.nrows) {
            const int rr = cur.row0 + r;
            const int t = p.q_list[cur.seg_off + rr / p.g];
            rows[j] = t * p.h_q + cur.h * p.g + rr % p.g;
          } else {
            rows[j] = oob_row;
          }
        }
#pragma unroll
        for (int cb = 0; cb < kCB; ++cb)
          tma_gather4(sQ0 + qs * L::kQ + cb * 128 * 128 + lane * 4 * 128, &tm_q, cb * 64, rows[0],
                      rows[1], rows[2], rows[3], &q_full[qs]);
      }
    }
  } else if (warp == 0) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0 && n > 0) {
      TileCursor cs, co;   // S stream runs two tiles ahead of the O stream
      cs.start(p, nb, t_begin);
      co.start(p, nb, t_begin);
      auto issue_s = [&](int i) {
        cs.set(p, t_begin + i);
        const int ks = cs.jseg % KVS, qs = i % QS;
        if (cs.new_seg) mbar_wait_sticky(&kv_full[ks], (cs.jseg / KVS) & 1, p.status, &fail);
        mbar_wait_sticky(&q_full[qs], (i / QS) & 1, p.status, &fail);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_f16(tS0 + (i & 1) * BK, desc_kmajor(sQ0 + qs * L::kQ, 128, kk),
                  desc_kmajor(sK0 + ks * L::kK, BK, kk), kIdescS, kk > 0);
        mma_commit(&s_full[i & 1]);
      };
      // S(i + 1) is issued ahead of O(i) unless its Q stage or K/V buffer is only
      // released by O(i) itself (single-buffered configurations).
      int next_s = 0;
      for (int i = 0; i < n; ++i) {
        if (next_s == i) issue_s(next_s++);
        if (next_s == i + 1 && i + 1 < n && QS >= 2 &&
            !(KVS == 1 && t_begin + i + 1 >= cs.seg_end_tile))
          issue_s(next_s++);
        co.set(p, t_begin + i);
        const int ks = co.jseg % KVS, ps = i % PS, os = i % OS;
        mbar_wait_sticky(&p_full[ps], (i / PS) & 1, p.status, &fail);
        if (i >= OS) mbar_wait_sticky(&o_free[os], ((i / OS) - 1) & 1, p.status, &fail);
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_f16(tO0 + os * D, desc_kmajor(sP0 + ps * L::kP, 128, kk),
                  desc_mnmajor(sV0 + ks * L::kK, BK, kk), kIdescO, kk > 0);
        mma_commit(&o_full[i & 1]);
        mma_commit(&p_empty[i & 1]);
        if (t_begin + i + 1 == co.seg_end_tile || i + 1 == n) mma_commit(&kv_empty[ks]);
      }
    }
  } else if (warp >= 4) {
    // ------------------------- softmax + epilogue -------------------------
    const int wg = (warp - 4) >> 2;
    const int row = tid - 128 - wg * 128;                  // tile row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    TileCursor cur;
    if (n > 0) cur.start(p, nb, t_begin);
    uint16_t *obuf = static_cast<uint16_t *>(p.obuf);
    for (int i = wg; i < n; i += 2) {
      cur.set(p, t_begin + i);
      const bool row_in = row < cur.nrows;
      int lim = -1;
      if (row_in) {
        const int t = p.q_list[cur.seg_off + (cur.row0 + row) / p.g];
        lim = min(BK - 1, t - cur.key0);
      }
      const int ps = i % PS, os = i % OS, qs = i % QS;
      mbar_wait_sticky(&s_full[i & 1], (i >> 1) & 1, p.status, &fail);
      tc_fence_after();
      const uint32_t tS = tS0 + (i & 1) * BK + lane_off;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BK / 32; ++c) {
        float sv[32];
        tmem_ld32(tS + c * 32, sv);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c * 32 + j <= lim) mx = fmaxf(mx, sv[j]);
      }
      const float m2 = row_in ? mx * p.scale_log2 : 0.f;
      // the P buffer is free once O of the previous tile that used it is done
      if (PS == 2 && i >= 2) mbar_wait_sticky(&p_empty[i & 1], ((i >> 1) - 1) & 1, p.status, &fail);
      if (PS == 1 && i >= 1)
        mbar_wait_sticky(&p_empty[(i - 1) & 1], ((i - 1) >> 1) & 1, p.status, &fail);
      float lsum = 0.f;
      const uint32_t sP = sP0 + ps * L::kP;
#pragma unroll
      for (int c = 0; c < BK / 32; ++c) {
        float sv[32];
        tmem_ld32(tS + c * 32, sv);
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int ii = c * 32 + j;
          const float p0 = (ii <= lim) ? ex2_approx(fmaf(sv[j], p.scale_log2, -m2)) : 0.f;
          const float p1 = (ii + 1 <= lim) ? ex2_approx(fmaf(sv[j + 1], p.scale_log2, -m2)) : 0.f;
          lsum += p0 + p1;                    // fp32 row sum (exact lse)
          pk[j / 2] = pack2<kFp16>(p0, p1);   // P rounded to 16 bits for the PV MMA
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t so = sw128_offset(row, c * 4 + q4, 128);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sP + so), "r"(pk[q4 * 4]),
                       "r"(pk[q4 * 4 + 1]), "r"(pk[q4 * 4 + 2]), "r"(pk[q4 * 4 + 3])
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[ps]);

      // epilogue: O(i) -> 16-bit, staged (swizzled) in this tile's Q stage, then
      // copied to the tile's contiguous compact-buffer rows with coalesced stores
      mbar_wait_sticky(&o_full[i & 1], (i >> 1) & 1, p.status, &fail);
      tc_fence_after();
      const uint32_t stage = sQ0 + qs * L::kQ;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        tmem_ld32(tO0 + os * D + c * 32 + lane_off, ov);
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) pk[j / 2] = pack2<kFp16>(ov[j], ov[j + 1]);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t so = sw128_offset(row, c * 4 + q4, 128);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(stage + so),
                       "r"(pk[q4 * 4]), "r"(pk[q4 * 4 + 1]), "r"(pk[q4 * 4 + 2]),
                       "r"(pk[q4 * 4 + 3])
                       : "memory");
        }
      }
      tc_fence_before();
      mbar_arrive(&o_free[os]);
      const int64_t grow0 = (int64_t)cur.seg_off * p.g + cur.row0;
      if (row_in) p.mlbuf[grow0 + row] = make_float2(m2, lsum);
      named_bar_sync(1 + wg, 128);
      constexpr int kRowChunks = D / 8;
      for (int idx = row; idx < cur.nrows * kRowChunks; idx += 128) {
        const int r = idx / kRowChunks, ch = idx - r * kRowChunks;
        uint4 val;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                     : "r"(stage + sw128_offset(r, ch, 128)));
        *reinterpret_cast<uint4 *>(obuf + (grow0 + r) * D + ch * 8) = val;
      }
      named_bar_sync(1 + wg, 128);
      if (row == 0) mbar_arrive(&q_empty[qs]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_base, L::kTmemCols);
}

// One warp per (token, query head): combine the <= T partials.
template <int D, bool kFp16>
__global__ void __launch_bounds__(256) fwd_merge_kernel(Params p) {
  constexpr int E = D / 32;   // elements per lane
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid >= (int64_t)p.n * p.h_q) return;
  const int t = static_cast<int>(wid / p.h_q), hq = static_cast<int>(wid - (int64_t)t * p.h_q);
  const int h = hq / p.g, j = hq - h * p.g;
  int64_t row = -1;
  if (lane < p.topk) {
    const int32_t pos = p.slot_map[((int64_t)h * p.n + t) * p.topk + lane];
    if (pos >= 0) row = (int64_t)pos * p.g + j;
  }
  float2 ml = make_float2(-INFINITY, 0.f);
  if (row >= 0) ml = p.mlbuf[row];
  float M = ml.x;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w = (row >= 0) ? ex2_approx(ml.x - M) : 0.f;
  float lsum = w * ml.y;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  const uint16_t *obuf = static_cast<const uint16_t *>(p.obuf);
  for (int kk = 0; kk < p.topk; ++kk) {
    const int64_t r = __shfl_sync(0xffffffffu, row, kk);
    const float wk = __shfl_sync(0xffffffffu, w, kk);
    if (r < 0) continue;
    const uint16_t *src = obuf + r * D + lane * E;
    uint32_t u[E / 2];
    if constexpr (E == 2) {
      u[0] = *reinterpret_cast<const uint32_t *>(src);
    } else if constexpr (E == 4) {
      const uint2 x = *reinterpret_cast<const uint2 *>(src);
      u[0] = x.x; u[1] = x.y;
    } else {
      const uint4 x = *reinterpret_cast<const uint4 *>(src);
      u[0] = x.x; u[1] = x.y; u[2] = x.z; u[3] = x.w;
    }
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
      const float2 f = unpack2<kFp16>(u[e]);
      acc[2 * e] = fmaf(wk, f.x, acc[2 * e]);
      acc[2 * e + 1] = fmaf(wk, f.y, acc[2 * e + 1]);
    }
  }
  const bool any = lsum > 0.f;
  const float inv = any ? 1.f / lsum : 0.f;
  uint32_t o[E / 2];
#pragma unroll
  for (int e = 0; e < E / 2; ++e) o[e] = pack2<kFp16>(acc[2 * e] * inv, acc[2 * e + 1] * inv);
  uint16_t *dst = static_cast<uint16_t *>(p.out) + ((int64_t)t * p.h_q + hq) * D + lane * E;
  if constexpr (E == 2) {
    *reinterpret_cast<uint32_t *>(dst) = o[0];
  } else if constexpr (E == 4) {
    *reinterpret_cast<uint2 *>(dst) = make_uint2(o[0], o[1]);
  } else {
    *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (lane == 0)
    p.lse[(int64_t)hq * p.n + t] = any ? (M + __log2f(lsum)) * 0.69314718055994531f : -INFINITY;
}

// ---------------------------------------------------------------------------
// Host-side dispatch
// ---------------------------------------------------------------------------
static bool encode_map(CUtensorMap *map, bool fp16, int rank, const void *base,
                       const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box) {
  using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static const EncodeFn encode = driver_entry<EncodeFn>("cuTensorMapEncodeTiled");
  if (!encode) return false;
  const cuuint32_t elem[3] = {1, 1, 1};
  return encode(map,
                                fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                rank, const_cast<void *>(base), dims, strides, box, elem,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of q ([N * h_q rows, d], one-row box for tile::gather4) and k, v
// ([N, h_k, d], box = B_K tokens x 1 head x 64 columns), 128-byte swizzle.
bool make_qkv_maps(const Params &p, const void *q, CUtensorMap *mq, CUtensorMap *mk,
                   CUtensorMap *mv) {
  const bool f16 = p.dtype == NSA_FP16;
  const cuuint64_t qdims[2] = {static_cast<cuuint64_t>(p.d),
                               static_cast<cuuint64_t>(p.n) * p.h_q};
  const cuuint64_t qstr[1] = {static_cast<cuuint64_t>(p.d) * 2};
  const cuuint32_t qbox[2] = {64, 1};
  const cuuint64_t kdims[3] = {static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.h_k),
                               static_cast<cuuint64_t>(p.n)};
  const cuuint64_t kstr[2] = {static_cast<cuuint64_t>(p.d) * 2,
                              static_cast<cuuint64_t>(p.h_k) * p.d * 2};
  const cuuint32_t kbox[3] = {64, 1, static_cast<cuuint32_t>(p.block)};
  return encode_map(mq, f16, 2, q, qdims, qstr, qbox) &&
         encode_map(mk, f16, 3, p.k, kdims, kstr, kbox) &&
         encode_map(mv, f16, 3, p.v, kdims, kstr, kbox);
}

template <int D, int BK, bool kFp16>
static cudaError_t run_fwd(const Params &p, int num_sms, int64_t max_tiles, cudaStream_t stream,
                           void (*mark)(int, cudaStream_t, bool)) {
  using L = FwdSmem<D, BK>;
  CUtensorMap mq, mk, mv;
  if (!make_qkv_maps(p, p.q, &mq, &mk, &mv)) return cudaErrorInvalidValue;
  // One CTA per SM: it owns all 512 TMEM columns.
  const uint32_t smem = L::kBytes > 120u * 1024u ? L::kBytes : 120u * 1024u;
  cudaError_t e = cudaFuncSetAttribute(fwd_main_kernel<D, BK, kFp16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int64_t grid = num_sms;
  if (grid > max_tiles) grid = max_tiles > 0 ? max_tiles : 1;
  mark(5, stream, true);
  fwd_main_kernel<D, BK, kFp16>
      <<<static_cast<unsigned>(grid), kFwdThreads, smem, stream>>>(mq, mk, mv, p);
  mark(5, stream, false);
  const int64_t rows = static_cast<int64_t>(p.n) * p.h_q;
  mark(6, stream, true);
  fwd_merge_kernel<D, kFp16><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(p);
  mark(6, stream, false);
  return cudaGetLastError();
}

template <int D, bool kFp16>
static cudaError_t run_fwd_bk(const Params &p, int num_sms, int64_t max_tiles, cudaStream_t s,
                              void (*mark)(int, cudaStream_t, bool)) {
  switch (p.block) {
    case 32: return run_fwd<D, 32, kFp16>(p, num_sms, max_tiles, s, mark);
    case 64: return run_fwd<D, 64, kFp16>(p, num_sms, max_tiles, s, mark);
    case 128: return run_fwd<D, 128, kFp16>(p, num_sms, max_tiles, s, mark);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fwd(const Params &p, int num_sms, int64_t max_tiles, cudaStream_t s,
                       void (*mark)(int, cudaStream_t, bool)) {
  const bool f16 = p.dtype == NSA_FP16;
  switch (p.d) {
    case 64: return f16 ? run_fwd_bk<64, true>(p, num_sms, max_tiles, s, mark)
                        : run_fwd_bk<64, false>(p, num_sms, max_tiles, s, mark);
    case 128: return f16 ? run_fwd_bk<128, true>(p, num_sms, max_tiles, s, mark)
                         : run_fwd_bk<128, false>(p, num_sms, max_tiles, s, mark);
    case 256: return f16 ? run_fwd_bk<256, true>(p, num_sms, max_tiles, s, mark)
                         : run_fwd_bk<256, false>(p, num_sms, max_tiles, s, mark);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nsa
