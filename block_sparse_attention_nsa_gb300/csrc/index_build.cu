// index_build.cu -- GPU index builder: selection tensor -> per-KV-block query
// lists (I_i) and per-(token, slot) compact-buffer positions (O_i), the index
// tensors of "FSA: An Alternative Efficient Implementation of Native Sparse
// Attention Kernel", key design 2.  It is a stable counting sort of the kept
// (token, slot) pairs by (KV head, global block):
//   geometry  -> per-sequence first global block, NB
//   count     -> per token-tile histogram over blocks (tile = kIdxWarps x 32 tokens)
//   col_scan  -> per block, exclusive prefix over token tiles, block totals
//   scan      -> exclusive prefix over (head, block): offsets, tile and chunk offsets
//   scatter   -> positions: block offset + earlier tiles + earlier warps + rank in warp
// Tokens inside a block's list come out ascending and duplicates keep their first
// slot, so the result is unique and bit-reproducible (no atomics decide order).
#include "common.cuh"

namespace nsa {

// ---------------------------------------------------------------------------
// geometry: blk_start[s] = sum_{s' < s} ceil(len_s' / B_K); nb = blk_start[S].
// A malformed cu_seqlens flags NSA_DEVERR_BAD_SEQLENS and yields nb = 0.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) geometry_kernel(Params p) {
  __shared__ int32_t warp_sums[32];
  __shared__ int bad;
  const int S = p.num_seqs, tid = threadIdx.x, nt = blockDim.x;
  if (tid == 0) bad = (p.cu[0] != 0 || p.cu[S] != p.n);
  __syncthreads();
  const int per = (S + nt - 1) / nt;
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
  int32_t local = 0;
  for (int s = s0; s < s1; ++s) {
    const int32_t len = p.cu[s + 1] - p.cu[s];
    if (len < 0) bad = 1;
    local += len > 0 ? (len + p.block - 1) / p.block : 0;
  }
  // block-wide exclusive scan of `local`
  const int lane = tid & 31, warp = tid >> 5;
  int32_t x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t w = lane < (nt >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  int32_t run = x - local + (warp > 0 ? warp_sums[warp - 1] : 0);
  for (int s = s0; s < s1; ++s) {
    p.blk_start[s] = run;
    const int32_t len = p.cu[s + 1] - p.cu[s];
    run += len > 0 ? (len + p.block - 1) / p.block : 0;
  }
  __syncthreads();
  if (tid == nt - 1) {
    const int32_t total = x + (warp > 0 ? warp_sums[warp - 1] : 0);
    p.blk_start[S] = total;
    if (bad) {
      set_status(p.status, NSA_DEVERR_BAD_SEQLENS);
      *p.nb = 0;
    } else {
      *p.nb = total;
    }
  }
}

// ---------------------------------------------------------------------------
// One pass over a warp's 32 tokens, in token order.  Lanes cover (token, slot)
// pairs: tokens_per_step = 32 / TP tokens per step, TP = next power of two >= T.
// kScatter = false: counts per block into bins (this warp's shared-memory row).
// kScatter = true : bins hold this warp's running base position per block; writes
//                   q_list and slot_map.
// ---------------------------------------------------------------------------
template <bool kScatter>
__device__ __forceinline__ void walk_tokens(const Params &p, int h, int tok0, int tok_end,
                                            int tp, int32_t *bins, int nb) {
  const int lane = threadIdx.x & 31;
  const int tps = 32 / tp;
  const int slot = lane & (tp - 1), sub = lane / tp;
  for (int base = tok0; base < tok_end; base += tps) {
    const int t = base + sub;
    const bool live = (slot < p.topk) && (t < tok_end);
    int32_t b = -1;
    int gb = -1;
    bool ok = false;
    if (live) {
      b = __ldg(p.sel + ((int64_t)h * p.n + t) * p.topk + slot);
      const int s = seq_of(p.cu, p.num_seqs, t);
      const int tau = t - p.cu[s];
      const int nblk = p.blk_start[s + 1] - p.blk_start[s];
      ok = (b >= 0) && (b <= tau / p.block) && (b < nblk);
      if (!kScatter && (b < -1 || b >= nblk)) set_status(p.status, NSA_DEVERR_BAD_INDEX);
      gb = p.blk_start[s] + b;
    }
    // duplicates inside one token: the lowest slot keeps the block
    const uint64_t key1 = ok ? ((static_cast<uint64_t>(sub) << 32) | static_cast<uint32_t>(b))
                             : (0xFFFFFFFF00000000ull | static_cast<uint64_t>(lane));
    const uint32_t m1 = __match_any_sync(0xffffffffu, key1);
    const bool keep = ok && ((__ffs(m1) - 1) == lane);
    // lanes of different tokens naming the same block (at most one lane per token)
    const uint32_t key2 = keep ? static_cast<uint32_t>(gb) : (0x80000000u | lane);
    const uint32_t m2 = __match_any_sync(0xffffffffu, key2);
    const bool leader = keep && ((__ffs(m2) - 1) == lane);
    if constexpr (!kScatter) {
      if (leader) bins[gb] += __popc(m2);
    } else {
      int32_t pos = -1;
      if (keep) pos = bins[gb] + __popc(m2 & ((1u << lane) - 1u));
      __syncwarp();
      if (leader) bins[gb] += __popc(m2);
      __syncwarp();
      if (live) {
        p.slot_map[((int64_t)h * p.n + t) * p.topk + slot] = pos;
        if (keep) p.q_list[pos] = t;
      }
    }
  }
  (void)nb;
}

// grid (n_idx_tiles, h_k), block idx_warps*32; dynamic smem idx_warps * nb_max ints
__global__ void __launch_bounds__(kIdxWarps * 32) count_kernel(Params p, int tp) {
  extern __shared__ int32_t bins_all[];
  const int nb = *p.nb;
  const int h = blockIdx.y, tile = blockIdx.x, W = p.idx_warps;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < W * nb; i += blockDim.x) bins_all[i] = 0;
  __syncthreads();
  const int tok0 = (tile * W + warp) * 32;
  if (tok0 < p.n) walk_tokens<false>(p, h, tok0, min(p.n, tok0 + 32), tp, bins_all + warp * nb, nb);
  __syncthreads();
  int32_t *hist = p.chunk_hist + ((int64_t)h * p.n_idx_tiles + tile) * p.nb_max;
  for (int gb = threadIdx.x; gb < nb; gb += blockDim.x) {
    int32_t s = 0;
    for (int w = 0; w < W; ++w) s += bins_all[w * nb + gb];
    hist[gb] = s;
  }
}

// grid (ceil(nb_max / 32), h_k), block (32, 8): exclusive prefix over token tiles
__global__ void __launch_bounds__(256) col_scan_kernel(Params p) {
  __shared__ int32_t part[8][33];
  const int nb = *p.nb;
  const int gb = blockIdx.x * 32 + threadIdx.x, h = blockIdx.y, y = threadIdx.y;
  const int64_t T = p.n_idx_tiles;
  const int64_t per = (T + 7) / 8;
  const int64_t t0 = min(T, y * per), t1 = min(T, t0 + per);
  int32_t *col = p.chunk_hist + (int64_t)h * T * p.nb_max + gb;
  int32_t local = 0;
  if (gb < nb)
    for (int64_t t = t0; t < t1; ++t) local += col[t * p.nb_max];
  part[y][threadIdx.x] = local;
  __syncthreads();
  int32_t run = 0;
  for (int yy = 0; yy < y; ++yy) run += part[yy][threadIdx.x];
  if (gb < nb) {
    for (int64_t t = t0; t < t1; ++t) {
      const int32_t c = col[t * p.nb_max];
      col[t * p.nb_max] = run;
      run += c;
    }
    if (y == 7) p.counts[h * nb + gb] = run;
  }
}

// One block of 1024 threads: offsets (pairs), tile_off (128-row tiles) and
// chunk_off (backward chunks of up to kBwdChunkTiles tiles) over h_k * nb segments.
__global__ void __launch_bounds__(1024) scan_kernel(Params p) {
  __shared__ int64_t sums[3][32];
  const int nseg = p.h_k * (*p.nb);
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nseg + nt - 1) / nt;
  const int i0 = min(nseg, tid * per), i1 = min(nseg, i0 + per);
  int64_t a = 0, b = 0, c = 0;
  for (int i = i0; i < i1; ++i) {
    const int64_t rows = (int64_t)p.counts[i] * p.g;
    const int64_t tiles = (rows + kTileRows - 1) / kTileRows;
    a += p.counts[i];
    b += tiles;
    c += (tiles + kBwdChunkTiles - 1) / kBwdChunkTiles;
  }
  int64_t xa = a, xb = b, xc = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int64_t ya = __shfl_up_sync(0xffffffffu, xa, o);
    int64_t yb = __shfl_up_sync(0xffffffffu, xb, o);
    int64_t yc = __shfl_up_sync(0xffffffffu, xc, o);
    if (lane >= o) { xa += ya; xb += yb; xc += yc; }
  }
  if (lane == 31) { sums[0][warp] = xa; sums[1][warp] = xb; sums[2][warp] = xc; }
  __syncthreads();
  if (warp == 0) {
    for (int k = 0; k < 3; ++k) {
      int64_t w = lane < (nt >> 5) ? sums[k][lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      sums[k][lane] = w;
    }
  }
  __syncthreads();
  int64_t ra = xa - a + (warp ? sums[0][warp - 1] : 0);
  int64_t rb = xb - b + (warp ? sums[1][warp - 1] : 0);
  int64_t rc = xc - c + (warp ? sums[2][warp - 1] : 0);
  for (int i = i0; i < i1; ++i) {
    p.offsets[i] = static_cast<int32_t>(ra);
    p.tile_off[i] = static_cast<int32_t>(rb);
    p.chunk_off[i] = static_cast<int32_t>(rc);
    const int64_t rows = (int64_t)p.counts[i] * p.g;
    const int64_t tiles = (rows + kTileRows - 1) / kTileRows;
    ra += p.counts[i];
    rb += tiles;
    rc += (tiles + kBwdChunkTiles - 1) / kBwdChunkTiles;
  }
  if (tid == nt - 1) {
    p.offsets[nseg] = static_cast<int32_t>(ra);
    p.tile_off[nseg] = static_cast<int32_t>(rb);
    p.chunk_off[nseg] = static_cast<int32_t>(rc);
  }
}

// Same grid as count_kernel.
__global__ void __launch_bounds__(kIdxWarps * 32) scatter_kernel(Params p, int tp) {
  extern __shared__ int32_t bins_all[];
  const int nb = *p.nb;
  const int h = blockIdx.y, tile = blockIdx.x, W = p.idx_warps;
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < W * nb; i += blockDim.x) bins_all[i] = 0;
  __syncthreads();
  const int tok0 = (tile * W + warp) * 32;
  const int tok1 = min(p.n, tok0 + 32);
  // status bits were raised by the count pass; only the per-warp counts are needed here
  if (tok0 < p.n) walk_tokens<false>(p, h, tok0, tok1, tp, bins_all + warp * nb, nb);
  __syncthreads();
  const int32_t *hist = p.chunk_hist + ((int64_t)h * p.n_idx_tiles + tile) * p.nb_max;
  for (int gb = threadIdx.x; gb < nb; gb += blockDim.x) {
    int32_t run = p.offsets[h * nb + gb] + hist[gb];
    for (int w = 0; w < W; ++w) {
      const int32_t c = bins_all[w * nb + gb];
      bins_all[w * nb + gb] = run;
      run += c;
    }
  }
  __syncthreads();
  if (tok0 < p.n) walk_tokens<true>(p, h, tok0, tok1, tp, bins_all + warp * nb, nb);
}

// ---------------------------------------------------------------------------
// Host launcher
// ---------------------------------------------------------------------------
cudaError_t launch_index(const Params &p, cudaStream_t stream, void (*mark)(int, cudaStream_t, bool)) {
  int tp = 1;
  while (tp < p.topk) tp <<= 1;
  mark(0, stream, true);
  geometry_kernel<<<1, 1024, 0, stream>>>(p);
  mark(0, stream, false);
  const size_t smem = sizeof(int32_t) * p.idx_warps * p.nb_max;
  dim3 grid_t(static_cast<unsigned>(p.n_idx_tiles), p.h_k);
  mark(1, stream, true);
  count_kernel<<<grid_t, p.idx_warps * 32, smem, stream>>>(p, tp);
  mark(1, stream, false);
  mark(2, stream, true);
  col_scan_kernel<<<dim3(static_cast<unsigned>((p.nb_max + 31) / 32), p.h_k), dim3(32, 8), 0,
                    stream>>>(p);
  mark(2, stream, false);
  mark(3, stream, true);
  scan_kernel<<<1, 1024, 0, stream>>>(p);
  mark(3, stream, false);
  mark(4, stream, true);
  scatter_kernel<<<grid_t, p.idx_warps * 32, smem, stream>>>(p, tp);
  mark(4, stream, false);
  return cudaGetLastError();
}

cudaError_t index_set_smem_limits(size_t smem) {
  cudaError_t e = cudaFuncSetAttribute(count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(smem));
}

}  // namespace nsa
