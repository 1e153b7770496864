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

template <int D, int BK>
struct FwdSmem {
  static constexpr int kPCols = BK < 64 ? 64 : BK;
  static constexpr uint32_t kQ = 128u * D * 2u;       // also the output staging tile
  static constexpr uint32_t kK = uint32_t(BK) * D * 2u;
  static constexpr uint32_t kP = 128u * kPCols * 2u;
  static constexpr uint32_t kOffQ = 0, kOffK = kQ, kOffV = kQ + kK, kOffP = kQ + 2 * kK;
  static constexpr uint32_t kBytes = kOffP + kP + 1024;   // + alignment slack
  static constexpr uint32_t kTmemCols = (128 + D) <= 256 ? 256 : 512;   // S at 0, O at 128
};

template <int D, int BK, bool kFp16>
__global__ void __launch_bounds__(kThreads, 1) fwd_main_kernel(Params p) {
  using L = FwdSmem<D, BK>;
  constexpr int kChunks = D / 8;                   // 16-byte chunks per row
  constexpr uint32_t kIdescS = idesc_f16(128, BK, false, false, kFp16);
  constexpr uint32_t kIdescO = idesc_f16(128, D, false, true, kFp16);

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + L::kOffQ), sK = smem_u32(smem + L::kOffK),
                 sV = smem_u32(smem + L::kOffV), sP = smem_u32(smem + L::kOffP);
  const int tid = threadIdx.x, warp = tid >> 5;

  if (warp == 0) tmem_alloc(&tmem_base, L::kTmemCols);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS = tmem_base, tO = tmem_base + 128;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  const int nb = *p.nb;
  const int nseg = p.h_k * nb;
  const int total_tiles = p.tile_off[nseg];
  const __nv_bfloat16 *gq = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *gk = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(p.v);
  uint16_t *obuf = static_cast<uint16_t *>(p.obuf);
  uint32_t phase = 0;
  int cur_seg = -1;

  for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
    const int seg = upper_index(p.tile_off, nseg + 1, tile);
    const int h = seg / nb, gb = seg - h * nb;
    const int s = upper_index(p.blk_start, p.num_seqs + 1, gb);
    const int b = gb - p.blk_start[s];
    const int key0 = p.cu[s] + b * BK;
    const int nkeys = min(BK, p.cu[s + 1] - key0);
    const int seg_off = p.offsets[seg];
    const int seg_rows = (p.offsets[seg + 1] - seg_off) * p.g;
    const int row0 = (tile - p.tile_off[seg]) * 128;
    const int nrows = min(128, seg_rows - row0);

    // ---- stage K_b, V_b (once per segment) and the gathered Q rows ----
    if (seg != cur_seg) {
      for (int idx = tid; idx < BK * kChunks; idx += kThreads) {
        const int r = idx / kChunks, ch = idx - r * kChunks;
        const bool in = r < nkeys;
        const int64_t off = in ? ((int64_t)(key0 + r) * p.h_k + h) * D + ch * 8 : 0;
        const uint32_t so = sw128_offset(r, ch, BK);
        cp_async16(sK + so, gk + off, in ? 16u : 0u);
        cp_async16(sV + so, gv + off, in ? 16u : 0u);
      }
      cur_seg = seg;
    }
    for (int idx = tid; idx < 128 * kChunks; idx += kThreads) {
      const int r = idx / kChunks, ch = idx - r * kChunks;
      const bool in = r < nrows;
      int64_t off = 0;
      if (in) {
        const int rr = row0 + r;
        const int t = p.q_list[seg_off + rr / p.g];
        const int hq = h * p.g + rr % p.g;
        off = ((int64_t)t * p.h_q + hq) * D + ch * 8;
      }
      cp_async16(sQ + sw128_offset(r, ch, 128), gq + off, in ? 16u : 0u);
    }
    cp_async_commit();
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncthreads();

    // ---- S = Q K_b^T ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        mma_f16(tS, desc_kmajor(sQ, 128, ks), desc_kmajor(sK, BK, ks), kIdescS, ks > 0);
      mma_commit(&bar);
    }
    bool ok = mbar_wait(&bar, phase, p.status);
    phase ^= 1;
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();

    // ---- row statistics and P (this thread owns tile row `tid` = TMEM lane) ----
    const bool row_in = tid < nrows;
    int lim = -1;   // last unmasked key of the block for this row
    if (row_in) {
      const int t = p.q_list[seg_off + (row0 + tid) / p.g];
      lim = min(BK - 1, t - key0);   // causal: key0 + i <= t
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < BK / 32; ++c) {
      float sv[32];
      tmem_ld32(tS + lane_off + c * 32, sv);
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c * 32 + j <= lim) mx = fmaxf(mx, sv[j]);
    }
    const float m2 = row_in ? mx * p.scale_log2 : 0.f;
    float lsum = 0.f;
#pragma unroll
    for (int c = 0; c < BK / 32; ++c) {
      float sv[32];
      tmem_ld32(tS + lane_off + c * 32, sv);
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) {
        const int i = c * 32 + j;
        const float p0 = (i <= lim) ? ex2_approx(fmaf(sv[j], p.scale_log2, -m2)) : 0.f;
        const float p1 = (i + 1 <= lim) ? ex2_approx(fmaf(sv[j + 1], p.scale_log2, -m2)) : 0.f;
        lsum += p0 + p1;                 // row sum of the fp32 values (exact lse)
        pk[j / 2] = pack2<kFp16>(p0, p1);   // P rounded to 16 bits for the PV MMA
      }
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t so = sw128_offset(tid, c * 4 + q4, 128);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sP + so), "r"(pk[q4 * 4]),
                     "r"(pk[q4 * 4 + 1]), "r"(pk[q4 * 4 + 2]), "r"(pk[q4 * 4 + 3])
                     : "memory");
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- O = P V_b ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < BK / 16; ++ks)
        mma_f16(tO, desc_kmajor(sP, 128, ks), desc_mnmajor(sV, BK, ks), kIdescO, ks > 0);
      mma_commit(&bar);
    }
    ok = mbar_wait(&bar, phase, p.status);
    phase ^= 1;
    if (__syncthreads_or(!ok)) break;
    tc_fence_after();

    // ---- epilogue: O row -> 16-bit -> swizzled staging (Q tile) -> contiguous rows ----
    const int64_t grow0 = (int64_t)seg_off * p.g + row0;   // first compact-buffer row of the tile
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float ov[32];
      tmem_ld32(tO + lane_off + c * 32, ov);
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 32; j += 2) pk[j / 2] = pack2<kFp16>(ov[j], ov[j + 1]);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t so = sw128_offset(tid, c * 4 + q4, 128);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sQ + so), "r"(pk[q4 * 4]),
                     "r"(pk[q4 * 4 + 1]), "r"(pk[q4 * 4 + 2]), "r"(pk[q4 * 4 + 3])
                     : "memory");
      }
    }
    if (row_in) p.mlbuf[grow0 + tid] = make_float2(m2, lsum);
    tc_fence_before();
    __syncthreads();
    for (int idx = tid; idx < nrows * kChunks; idx += kThreads) {
      const int r = idx / kChunks, ch = idx - r * kChunks;
      uint4 val;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                   : "r"(sQ + sw128_offset(r, ch, 128)));
      *reinterpret_cast<uint4 *>(obuf + (grow0 + r) * D + ch * 8) = val;
    }
    __syncthreads();
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
template <int D, int BK, bool kFp16>
static cudaError_t run_fwd(const Params &p, int num_sms, int64_t max_tiles, cudaStream_t stream,
                           void (*mark)(int, cudaStream_t, bool)) {
  using L = FwdSmem<D, BK>;
  const int per_sm = 512 / L::kTmemCols;
  // Request enough shared memory that no more CTAs share an SM than TMEM allows.
  const uint32_t floor_bytes = per_sm == 1 ? 120u * 1024u : 80u * 1024u;
  const uint32_t smem = L::kBytes > floor_bytes ? L::kBytes : floor_bytes;
  cudaError_t e = cudaFuncSetAttribute(fwd_main_kernel<D, BK, kFp16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int64_t grid = static_cast<int64_t>(num_sms) * per_sm;
  if (grid > max_tiles) grid = max_tiles > 0 ? max_tiles : 1;
  mark(5, stream, true);
  fwd_main_kernel<D, BK, kFp16><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(p);
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
