// bwd.cu -- backward of NSA selected attention on sm_103a.
//
// Same KV-block-outer order as the forward ("FSA: An Alternative Efficient
// Implementation of Native Sparse Attention Kernel", key designs 1-2; the
// backward reuses the forward's index tensors I_i / O_i):
//
//   bwd_pre   : D[hq, t] = sum_d dO * O  (fp32).
//   bwd_main  : one CTA per chunk of <= kBwdChunkTiles row tiles of one
//               (KV head, block) segment.  Per tile, on tcgen05 with TMEM
//               accumulators:  S = Q K_b^T and dP = dO V_b^T;  in registers
//               P = exp2(S*scale*log2e - lse*log2e) (causal mask), dS = P (dP - D);
//               dV_b^T += dO^T P and dK_b^T += Q^T dS stay in TMEM across the
//               chunk; dQ_part = dS K_b goes to the compact buffer at the pair's
//               position.  At the end of the chunk dK_b, dV_b partials are written
//               per chunk (no atomics).
//   bwd_dq    : per (token, query head), dq = scale * sum of its <= T dQ partials.
//   bwd_dkv   : per (KV head, block), dk = scale * sum of chunk partials of dK,
//               dv = sum of those of dV; blocks nobody selected get zeros.
#include "common.cuh"

namespace nsa {

__device__ __forceinline__ float ex2_approx_b(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// D = rowsum(dO * O): one warp per (token, query head)
// ---------------------------------------------------------------------------
template <int D, bool kFp16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(Params p) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid >= (int64_t)p.n * p.h_q) return;
  const int t = static_cast<int>(wid / p.h_q), hq = static_cast<int>(wid - (int64_t)t * p.h_q);
  const uint16_t *o = static_cast<const uint16_t *>(p.out_in) + wid * D + lane * E;
  const uint16_t *g = static_cast<const uint16_t *>(p.dout) + wid * D + lane * E;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const float2 a = unpack2<kFp16>(*reinterpret_cast<const uint32_t *>(o + e));
    const float2 b = unpack2<kFp16>(*reinterpret_cast<const uint32_t *>(g + e));
    acc = fmaf(a.x, b.x, fmaf(a.y, b.y, acc));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) p.dstat[(int64_t)hq * p.n + t] = acc;
}

template <int D, int BK>
struct BwdSmem {
  static constexpr int kPCols = BK < 64 ? 64 : BK;
  static constexpr uint32_t kQ = 128u * D * 2u;
  static constexpr uint32_t kK = uint32_t(BK) * D * 2u;
  static constexpr uint32_t kP = 128u * kPCols * 2u;
  static constexpr uint32_t kOffQ = 0, kOffDO = kQ, kOffK = 2 * kQ, kOffV = 2 * kQ + kK,
                            kOffP = 2 * kQ + 2 * kK, kOffDS = 2 * kQ + 2 * kK + kP;
  static constexpr uint32_t kBytes = kOffDS + kP + 1024;
  // TMEM: [0, R0) holds S, dP, later dQ; then dV^T, dK^T (BK columns each)
  // dV^T / dK^T use N = max(B_K, 64): one full 128-byte swizzle atom of P / dS columns
  static constexpr int kNKV = BK < 64 ? 64 : BK;
  static constexpr int kR0 = (2 * BK) > D ? (2 * BK) : D;
  static constexpr int kUsed = kR0 + 2 * kNKV;
  static constexpr uint32_t kTmemCols = kUsed <= 128 ? 128 : (kUsed <= 256 ? 256 : 512);
};

template <bool kFp16>
__device__ __forceinline__ void store_row_chunks(uint32_t tile, int row, int chunk0,
                                                 const float *vals32) {
  uint32_t pk[16];
#pragma unroll
  for (int j = 0; j < 32; j += 2) pk[j / 2] = pack2<kFp16>(vals32[j], vals32[j + 1]);
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint32_t so = sw128_offset(row, chunk0 + q4, 128);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tile + so), "r"(pk[q4 * 4]),
                 "r"(pk[q4 * 4 + 1]), "r"(pk[q4 * 4 + 2]), "r"(pk[q4 * 4 + 3])
                 : "memory");
  }
}

template <int D, int BK, bool kFp16>
__global__ void __launch_bounds__(kThreads, 1) bwd_main_kernel(Params p) {
  using L = BwdSmem<D, BK>;
  static_assert(D == 128, "backward main kernel: d = 128 (tcgen05 M = d for dK^T / dV^T)");
  static_assert(BK == 32 || BK == 64 || BK == 128, "block size");
  constexpr int kChunks = D / 8;
  constexpr uint32_t kIdescS = idesc_f16(128, BK, false, false, kFp16);     // S, dP
  constexpr uint32_t kIdescKV = idesc_f16(D, L::kNKV, true, true, kFp16);  // dV^T, dK^T
  constexpr uint32_t kIdescQ = idesc_f16(128, D, false, true, kFp16);      // dQ

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + L::kOffQ), sDO = smem_u32(smem + L::kOffDO),
                 sK = smem_u32(smem + L::kOffK), sV = smem_u32(smem + L::kOffV),
                 sP = smem_u32(smem + L::kOffP), sDS = smem_u32(smem + L::kOffDS);
  const int tid = threadIdx.x, warp = tid >> 5;

  if (warp == 0) tmem_alloc(&tmem_base, L::kTmemCols);
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS = tmem_base, tdP = tmem_base + BK, tdQ = tmem_base,
                 tdV = tmem_base + L::kR0, tdK = tmem_base + L::kR0 + L::kNKV;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  const int nb = *p.nb;
  const int nseg = p.h_k * nb;
  const int total_chunks = p.chunk_off[nseg];
  const __nv_bfloat16 *gq = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *gk = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *gv = static_cast<const __nv_bfloat16 *>(p.v);
  const __nv_bfloat16 *gdo = static_cast<const __nv_bfloat16 *>(p.dout);
  uint16_t *dqbuf = reinterpret_cast<uint16_t *>(p.dqbuf);
  const float kLog2e = 1.4426950408889634f;
  uint32_t phase = 0;
  bool failed = false;

  for (int chunk = blockIdx.x; chunk < total_chunks && !failed; chunk += gridDim.x) {
    const int seg = upper_index(p.chunk_off, nseg + 1, chunk);
    const int h = seg / nb, gb = seg - h * nb;
    const int s = upper_index(p.blk_start, p.num_seqs + 1, gb);
    const int b = gb - p.blk_start[s];
    const int key0 = p.cu[s] + b * BK;
    const int nkeys = min(BK, p.cu[s + 1] - key0);
    const int seg_off = p.offsets[seg];
    const int seg_rows = (p.offsets[seg + 1] - seg_off) * p.g;
    const int ntiles_seg = p.tile_off[seg + 1] - p.tile_off[seg];
    const int tile_begin = (chunk - p.chunk_off[seg]) * kBwdChunkTiles;
    const int tile_end = min(ntiles_seg, tile_begin + kBwdChunkTiles);

    // K_b, V_b for this chunk
    for (int idx = tid; idx < BK * kChunks; idx += kThreads) {
      const int r = idx / kChunks, ch = idx - r * kChunks;
      const bool in = r < nkeys;
      const int64_t off = in ? ((int64_t)(key0 + r) * p.h_k + h) * D + ch * 8 : 0;
      const uint32_t so = sw128_offset(r, ch, BK);
      cp_async16(sK + so, gk + off, in ? 16u : 0u);
      cp_async16(sV + so, gv + off, in ? 16u : 0u);
    }

    for (int tile = tile_begin; tile < tile_end; ++tile) {
      const int row0 = tile * 128;
      const int nrows = min(128, seg_rows - row0);
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
        const uint32_t so = sw128_offset(r, ch, 128);
        cp_async16(sQ + so, gq + off, in ? 16u : 0u);
        cp_async16(sDO + so, gdo + off, in ? 16u : 0u);
      }
      cp_async_commit();
      // per-row statistics (this thread's row)
      const bool row_in = tid < nrows;
      int lim = -1;
      float lse2 = 0.f, dval = 0.f;
      if (row_in) {
        const int rr = row0 + tid;
        const int t = p.q_list[seg_off + rr / p.g];
        const int hq = h * p.g + rr % p.g;
        lim = min(BK - 1, t - key0);
        lse2 = p.lse_in[(int64_t)hq * p.n + t] * kLog2e;
        dval = p.dstat[(int64_t)hq * p.n + t];
      }
      cp_async_wait_all();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();

      // S = Q K^T, dP = dO V^T
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_f16(tS, desc_kmajor(sQ, 128, ks), desc_kmajor(sK, BK, ks), kIdescS, ks > 0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          mma_f16(tdP, desc_kmajor(sDO, 128, ks), desc_kmajor(sV, BK, ks), kIdescS, ks > 0);
        mma_commit(&bar);
      }
      bool ok = mbar_wait(&bar, phase, p.status);
      phase ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; break; }
      tc_fence_after();

      // P and dS rows
#pragma unroll
      for (int c = 0; c < BK / 32; ++c) {
        float sv[32], dp[32];
        tmem_ld32(tS + lane_off + c * 32, sv);
        tmem_ld32(tdP + lane_off + c * 32, dp);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int i = c * 32 + j;
          float pr = (i <= lim) ? ex2_approx_b(fmaf(sv[j], p.scale_log2, -lse2)) : 0.f;
          pr = round16<kFp16>(pr);
          sv[j] = pr;
          dp[j] = pr * (dp[j] - dval);
        }
        store_row_chunks<kFp16>(sP, tid, c * 4, sv);
        store_row_chunks<kFp16>(sDS, tid, c * 4, dp);
      }
      if constexpr (BK < 64) {   // zero the unused half of the swizzle atom read by N = 64
        float z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0.f;
        store_row_chunks<kFp16>(sP, tid, 4, z);
        store_row_chunks<kFp16>(sDS, tid, 4, z);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();

      // dV^T += dO^T P, dK^T += Q^T dS (M = d), dQ = dS K (M = rows)
      if (tid == 0) {
        tc_fence_after();
        const bool first = (tile == tile_begin);
#pragma unroll
        for (int ks = 0; ks < 128 / 16; ++ks)
          mma_f16(tdV, desc_mnmajor(sDO, 128, ks), desc_mnmajor(sP, 128, ks), kIdescKV,
                  (!first || ks > 0) ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 128 / 16; ++ks)
          mma_f16(tdK, desc_mnmajor(sQ, 128, ks), desc_mnmajor(sDS, 128, ks), kIdescKV,
                  (!first || ks > 0) ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < BK / 16; ++ks)
          mma_f16(tdQ, desc_kmajor(sDS, 128, ks), desc_mnmajor(sK, BK, ks), kIdescQ, ks > 0);
        mma_commit(&bar);
      }
      ok = mbar_wait(&bar, phase, p.status);
      phase ^= 1;
      if (__syncthreads_or(!ok)) { failed = true; break; }
      tc_fence_after();

      // dQ partial rows -> 16-bit staging (Q tile) -> contiguous compact-buffer rows
      const int64_t grow0 = (int64_t)seg_off * p.g + row0;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tmem_ld32(tdQ + lane_off + c * 32, v);
        store_row_chunks<kFp16>(sQ, tid, c * 4, v);
      }
      tc_fence_before();
      __syncthreads();
      for (int idx = tid; idx < nrows * kChunks; idx += kThreads) {
        const int r = idx / kChunks, ch = idx - r * kChunks;
        uint4 val;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                     : "r"(sQ + sw128_offset(r, ch, 128)));
        *reinterpret_cast<uint4 *>(dqbuf + (grow0 + r) * D + ch * 8) = val;
      }
      __syncthreads();
    }
    if (failed) break;

    // chunk partials of dV, dK: TMEM lane = d index, column = key
    float *dst = p.dkvbuf + (int64_t)chunk * 2 * BK * D;
#pragma unroll
    for (int c = 0; c < BK / 32; ++c) {
      float v[32];
      tmem_ld32(tdV + lane_off + c * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) dst[(c * 32 + j) * D + tid] = v[j];
      tmem_ld32(tdK + lane_off + c * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) dst[(int64_t)BK * D + (c * 32 + j) * D + tid] = v[j];
    }
    tc_fence_before();
    __syncthreads();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem_base, L::kTmemCols);
}

// dq[t, hq] = scale * sum_k dQ_part[slot_map[h, t, k] * g + j]; one warp per row.
template <int D, bool kFp16>
__global__ void __launch_bounds__(256) bwd_dq_kernel(Params p) {
  constexpr int E = D / 32;
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
  const uint16_t *buf = reinterpret_cast<const uint16_t *>(p.dqbuf);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int kk = 0; kk < p.topk; ++kk) {
    const int64_t r = __shfl_sync(0xffffffffu, row, kk);
    if (r < 0) continue;
    const uint16_t *src = buf + r * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 f = unpack2<kFp16>(*reinterpret_cast<const uint32_t *>(src + e));
      acc[e] += f.x;
      acc[e + 1] += f.y;
    }
  }
  uint16_t *dst = static_cast<uint16_t *>(p.dq) + wid * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    *reinterpret_cast<uint32_t *>(dst + e) = pack2<kFp16>(acc[e] * p.scale, acc[e + 1] * p.scale);
}

// dk, dv of one (KV head, block): sum over the segment's chunks (zeros if none).
template <int D, int BK, bool kFp16>
__global__ void __launch_bounds__(256) bwd_dkv_kernel(Params p) {
  const int nb = *p.nb;
  const int seg = blockIdx.x;
  if (seg >= p.h_k * nb) return;
  const int h = seg / nb, gb = seg - h * nb;
  const int s = upper_index(p.blk_start, p.num_seqs + 1, gb);
  const int b = gb - p.blk_start[s];
  const int key0 = p.cu[s] + b * BK;
  const int nkeys = min(BK, p.cu[s + 1] - key0);
  const int c0 = p.chunk_off[seg], c1 = p.chunk_off[seg + 1];
  uint16_t *dk = static_cast<uint16_t *>(p.dk), *dv = static_cast<uint16_t *>(p.dv);
  for (int idx = threadIdx.x * 2; idx < nkeys * D; idx += blockDim.x * 2) {
    const int key = idx / D, x = idx - key * D;
    float ak0 = 0.f, ak1 = 0.f, av0 = 0.f, av1 = 0.f;
    for (int c = c0; c < c1; ++c) {
      const float *src = p.dkvbuf + (int64_t)c * 2 * BK * D;
      const float2 v2 = *reinterpret_cast<const float2 *>(src + key * D + x);
      const float2 k2 = *reinterpret_cast<const float2 *>(src + BK * D + key * D + x);
      av0 += v2.x; av1 += v2.y; ak0 += k2.x; ak1 += k2.y;
    }
    const int64_t o = ((int64_t)(key0 + key) * p.h_k + h) * D + x;
    *reinterpret_cast<uint32_t *>(dk + o) = pack2<kFp16>(ak0 * p.scale, ak1 * p.scale);
    *reinterpret_cast<uint32_t *>(dv + o) = pack2<kFp16>(av0, av1);
  }
}

// ---------------------------------------------------------------------------
// Host-side dispatch
// ---------------------------------------------------------------------------
template <int D, int BK, bool kFp16>
static cudaError_t run_bwd(const Params &p, int num_sms, int64_t max_chunks, cudaStream_t stream,
                           void (*mark)(int, cudaStream_t, bool)) {
  using L = BwdSmem<D, BK>;
  const int64_t rows = static_cast<int64_t>(p.n) * p.h_q;
  mark(7, stream, true);
  bwd_pre_kernel<D, kFp16><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(p);
  mark(7, stream, false);
  const uint32_t smem = L::kBytes;
  cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel<D, BK, kFp16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int per_sm_tmem = 512 / L::kTmemCols;
  const int per_sm_smem = static_cast<int>((228u * 1024u) / (smem + 1024u));
  const int per_sm = per_sm_tmem < per_sm_smem ? per_sm_tmem : per_sm_smem;
  int64_t grid = static_cast<int64_t>(num_sms) * (per_sm > 0 ? per_sm : 1);
  if (grid > max_chunks) grid = max_chunks > 0 ? max_chunks : 1;
  mark(8, stream, true);
  bwd_main_kernel<D, BK, kFp16><<<static_cast<unsigned>(grid), kThreads, smem, stream>>>(p);
  mark(8, stream, false);
  mark(9, stream, true);
  bwd_dq_kernel<D, kFp16><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(p);
  mark(9, stream, false);
  mark(10, stream, true);
  bwd_dkv_kernel<D, BK, kFp16><<<static_cast<unsigned>(p.h_k * p.nb_max), 256, 0, stream>>>(p);
  mark(10, stream, false);
  return cudaGetLastError();
}

template <bool kFp16>
static cudaError_t run_bwd_bk(const Params &p, int num_sms, int64_t max_chunks, cudaStream_t s,
                              void (*mark)(int, cudaStream_t, bool)) {
  switch (p.block) {
    case 32: return run_bwd<128, 32, kFp16>(p, num_sms, max_chunks, s, mark);
    case 64: return run_bwd<128, 64, kFp16>(p, num_sms, max_chunks, s, mark);
    case 128: return run_bwd<128, 128, kFp16>(p, num_sms, max_chunks, s, mark);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd(const Params &p, int num_sms, int64_t max_chunks, cudaStream_t s,
                       void (*mark)(int, cudaStream_t, bool)) {
  if (p.d != 128) return cudaErrorInvalidValue;
  return p.dtype == NSA_FP16 ? run_bwd_bk<true>(p, num_sms, max_chunks, s, mark)
                             : run_bwd_bk<false>(p, num_sms, max_chunks, s, mark);
}

}  // namespace nsa
