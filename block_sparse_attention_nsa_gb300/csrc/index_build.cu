// index_build.cu -- GPU index builder: selection tensor -> per-KV-block query
// lists (I_i) and per-(token, slot) compact-buffer positions (O_i), the index
// tensors of "FSA: An Alternative Efficient Implementation of Native Sparse
// Attention Kernel", key design 2.  It is a stable counting sort of the kept
// (token, slot) pairs by (KV head, global block):
//   geometry   -> per-sequence first global block, NB
//   count      -> per token-tile histogram over blocks, kept pairs per token
//   col_scan   -> per block, exclusive prefix over token tiles, block totals
//   scan       -> exclusive prefix over (head, block): offsets, tile and chunk offsets
//   wave_scan  -> forward tiles of every (head, wave, block) sub-segment, prefix
//   tile_desc  -> one descriptor per forward tile
//   scatter    -> positions: block offset + earlier tiles + rank inside the tile
// Tokens inside a block's list come out ascending and duplicates keep their first
// slot, so the result is unique and bit-reproducible: ranks come from per-block
// token bitmasks (population counts), not from the order of atomic operations.
//
// One thread handles one token: it reads the token's T slots, drops invalid and
// repeated values in registers, and names each kept block once.
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
// The kept blocks of token t for KV head h: kgb[k] = global block of slot k, or
// -1 when slot k is empty, out of range, in the future, or repeats an earlier
// slot.  Returns the number of kept slots; raises *bad for values below -1 or
// past the sequence's last block.  TP = T rounded up to a power of two.
// ---------------------------------------------------------------------------
template <int TP>
__device__ __forceinline__ int token_blocks(const Params &p, int nb, int h, int t,
                                            int32_t (&kgb)[TP], bool &bad) {
  const int s = seq_of(p.cu, p.num_seqs, t);
  const int tau = t - __ldg(p.cu + s);
  const int c = tau / p.block;
  const int bs = p.blk_start[s];
  const int nblk = p.blk_start[s + 1] - bs;
  const int32_t *row = p.sel + ((int64_t)h * p.n + t) * p.topk;
  int np = 0;
#pragma unroll
  for (int k = 0; k < TP; ++k) {
    const bool in = k < p.topk;
    const int b = in ? __ldg(row + k) : -1;
    if (in && (b < -1 || b >= nblk)) bad = true;
    bool ok = in && b >= 0 && b <= c && b < nblk && bs + b < nb;
#pragma unroll
    for (int j = 0; j < k; ++j) ok = ok && (kgb[j] != bs + b);
    kgb[k] = ok ? bs + b : -1;
    np += ok ? 1 : 0;
  }
  return np;
}

// grid (n_idx_tiles, h_k), block kIdxThreads; dynamic smem nb_max ints.
// chunk_hist[h][tile][gb] = kept pairs of the tile's tokens naming block gb;
// npairs[h][t] = kept pairs of token t.
template <int TP>
__global__ void __launch_bounds__(kIdxThreads) count_kernel(Params p) {
  extern __shared__ int32_t bins[];
  const int nb = *p.nb;
  const int h = blockIdx.y, tile = blockIdx.x, tid = threadIdx.x;
  for (int i = tid; i < nb; i += blockDim.x) bins[i] = 0;
  __syncthreads();
  const int t = tile * p.idx_tok + tid;
  int32_t kgb[TP];
#pragma unroll
  for (int k = 0; k < TP; ++k) kgb[k] = -1;
  if (tid < p.idx_tok && t < p.n) {
    bool bad = false;
    int np = 0;
    if (nb > 0) {
      np = token_blocks<TP>(p, nb, h, t, kgb, bad);
    }
    if (bad) set_status(p.status, NSA_DEVERR_BAD_INDEX);
    p.npairs[(int64_t)h * p.n + t] = np;
  }
  {
    // lanes naming the same block as their warp's lowest active lane in slot k
    // (the own block and block 0, typically) add once for all of them
    const bool live = tid < p.idx_tok && t < p.n && nb > 0;
    const uint32_t act = __ballot_sync(0xffffffffu, live);
    if (live) {
      const int leader = __ffs(act) - 1;
#pragma unroll
      for (int k = 0; k < TP; ++k) {
        const int32_t lead_gb = __shfl_sync(act, kgb[k], leader);
        const uint32_t same = __ballot_sync(act, kgb[k] == lead_gb && kgb[k] >= 0);
        if (kgb[k] >= 0) {
          if (kgb[k] != lead_gb) atomicAdd(&bins[kgb[k]], 1);
          else if ((tid & 31) == leader) atomicAdd(&bins[kgb[k]], __popc(same));
        }
      }
    }
  }
  __syncthreads();
  int32_t *hist = p.chunk_hist + ((int64_t)h * p.n_idx_tiles + tile) * p.nb_max;
  for (int gb = tid; gb < nb; gb += blockDim.x) hist[gb] = bins[gb];
}

// grid (ceil(nb_max / 32), h_k), block (32, 32): exclusive prefix over token tiles;
// thread (x, y) covers block 32 * blockIdx.x + x and one range of token tiles.
__global__ void __launch_bounds__(1024) col_scan_kernel(Params p) {
  __shared__ int32_t part[32][33];
  const int nb = *p.nb;
  const int gb = blockIdx.x * 32 + threadIdx.x, h = blockIdx.y, y = threadIdx.y;
  const int64_t T = p.n_idx_tiles;
  const int64_t per = (T + 31) / 32;
  const int64_t t0 = min(T, y * per), t1 = min(T, t0 + per);
  int32_t *col = p.chunk_hist + (int64_t)h * T * p.nb_max + gb;
  int32_t local = 0;
  if (gb < nb) {
#pragma unroll 8
    for (int64_t t = t0; t < t1; ++t) local += col[t * p.nb_max];
  }
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
    if (y == 31) p.counts[h * nb + gb] = run;
  }
}

// One block of 1024 threads: offsets (pairs) and tile_off (128-row tiles) over the
// h_k * nb segments.  With a single forward wave the sub-segments are the segments,
// and wtile_off (indexed h * nb_max + block) is written here too.
__global__ void __launch_bounds__(1024) scan_kernel(Params p) {
  __shared__ int64_t sums[2][32];
  const int nseg = p.h_k * (*p.nb);
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int per = (nseg + nt - 1) / nt;
  const int i0 = min(nseg, tid * per), i1 = min(nseg, i0 + per);
  int64_t a = 0, b = 0;
  for (int i = i0; i < i1; ++i) {
    const int64_t rows = (int64_t)p.counts[i] * p.g;
    a += p.counts[i];
    b += (rows + kTileRows - 1) / kTileRows;
  }
  int64_t xa = a, xb = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int64_t ya = __shfl_up_sync(0xffffffffu, xa, o);
    int64_t yb = __shfl_up_sync(0xffffffffu, xb, o);
    if (lane >= o) { xa += ya; xb += yb; }
  }
  if (lane == 31) { sums[0][warp] = xa; sums[1][warp] = xb; }
  __syncthreads();
  if (warp == 0) {
    for (int k = 0; k < 2; ++k) {
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
  const int nb = *p.nb;
  for (int i = i0; i < i1; ++i) {
    p.offsets[i] = static_cast<int32_t>(ra);
    p.tile_off[i] = static_cast<int32_t>(rb);
    if (p.n_w == 1) p.wtile_off[(int64_t)(i / nb) * p.nb_max + i % nb] = static_cast<int32_t>(rb);
    const int64_t rows = (int64_t)p.counts[i] * p.g;
    ra += p.counts[i];
    rb += (rows + kTileRows - 1) / kTileRows;
  }
  if (tid == nt - 1) {
    p.offsets[nseg] = static_cast<int32_t>(ra);
    p.tile_off[nseg] = static_cast<int32_t>(rb);
  }
  if (p.n_w == 1) {
    // sub-segments of blocks nb .. nb_max - 1 hold no tiles: they start where the
    // next head's (or, for the last head, the grand total) does
    __syncthreads();
    const int64_t pad = p.nb_max - nb;
    for (int64_t e = tid; e < (int64_t)p.h_k * pad; e += nt) {
      const int h = static_cast<int>(e / pad), gb = nb + static_cast<int>(e % pad);
      p.wtile_off[(int64_t)h * p.nb_max + gb] = p.tile_off[(h + 1) * nb];
    }
    if (tid == 0) p.wtile_off[p.nsub] = p.tile_off[nseg];
  }
}

// ---------------------------------------------------------------------------
// Forward sub-segments.  Wave w covers index token tiles [w * wave_tiles,
// (w + 1) * wave_tiles); the tokens of wave w that selected block gb are a
// contiguous run of the block's ascending list I_gb, starting at the exclusive
// prefix chunk_hist[h][w * wave_tiles][gb].  Sub-segment id:
// (h * n_w + w) * nb_max + gb.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int32_t wave_lo(const Params &p, int nb, int h, int w, int gb) {
  const int64_t tile = (int64_t)w * p.wave_tiles;
  if (tile >= p.n_idx_tiles) return p.counts[h * nb + gb];
  return p.chunk_hist[((int64_t)h * p.n_idx_tiles + tile) * p.nb_max + gb];
}

__device__ __forceinline__ void sub_decode(const Params &p, int64_t i, int &h, int &w, int &gb) {
  gb = static_cast<int>(i % p.nb_max);
  const int64_t hw = i / p.nb_max;
  w = static_cast<int>(hw % p.n_w);
  h = static_cast<int>(hw / p.n_w);
}

// Rows of sub-segment i and its first list index (lo); 0 rows for blocks >= nb.
__device__ __forceinline__ int64_t sub_rows(const Params &p, int nb, int64_t i, int32_t *lo_out) {
  int h, w, gb;
  sub_decode(p, i, h, w, gb);
  if (gb >= nb) {
    *lo_out = 0;
    return 0;
  }
  const int32_t lo = wave_lo(p, nb, h, w, gb), hi = wave_lo(p, nb, h, w + 1, gb);
  *lo_out = lo;
  return (int64_t)(hi - lo) * p.g;
}

// Multi-CTA exclusive scan of the forward tiles per sub-segment: each CTA of
// 1024 threads scans kScanPer entries locally and records its total.
__global__ void __launch_bounds__(1024) wave_scan_local_kernel(Params p) {
  __shared__ int32_t sums[32];
  constexpr int kPer = kScanPer / 1024;
  const int nb = *p.nb;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t base = (int64_t)blockIdx.x * kScanPer + (int64_t)tid * kPer;
  int32_t v[kPer];
  int32_t local = 0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int64_t i = base + e;
    int32_t lo;
    const int64_t rows = i < p.nsub ? sub_rows(p, nb, i, &lo) : 0;
    v[e] = static_cast<int32_t>((rows + kTileRows - 1) / kTileRows);
    local += v[e];
  }
  int32_t x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int32_t w = sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sums[lane] = w;
  }
  __syncthreads();
  int32_t run = x - local + (warp > 0 ? sums[warp - 1] : 0);
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int64_t i = base + e;
    if (i < p.nsub) p.wtile_off[i] = run;
    run += v[e];
  }
  if (tid == 1023) p.wscan_part[blockIdx.x] = sums[31];
}

// Adds the totals of earlier CTAs; the last CTA also writes the grand total.
__global__ void __launch_bounds__(1024) wave_scan_add_kernel(Params p) {
  __shared__ int32_t base_s;
  const int tid = threadIdx.x;
  if (tid < 32) {
    int32_t s = 0;
    for (int64_t c = tid; c < blockIdx.x; c += 32) s += p.wscan_part[c];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (tid == 0) base_s = s;
  }
  __syncthreads();
  const int32_t b = base_s;
  const int64_t i0 = (int64_t)blockIdx.x * kScanPer;
  for (int e = tid; e < kScanPer; e += 1024) {
    const int64_t i = i0 + e;
    if (i < p.nsub) p.wtile_off[i] += b;
  }
  if (blockIdx.x == gridDim.x - 1 && tid == 0)
    p.wtile_off[p.nsub] = b + p.wscan_part[blockIdx.x];
}

// One warp per sub-segment: lane j writes the descriptors of tiles j, j + 32, ...
__global__ void __launch_bounds__(256) tile_desc_kernel(Params p) {
  const int nb = *p.nb;
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (i >= p.nsub) return;
  const int32_t t0 = p.wtile_off[i], nt = p.wtile_off[i + 1] - t0;
  if (nt <= 0) return;
  int h, w, gb;
  sub_decode(p, i, h, w, gb);
  int32_t lo;
  const int64_t rows = sub_rows(p, nb, i, &lo);
  const int s = upper_index(p.blk_start, p.num_seqs + 1, gb);
  const int32_t key0 = p.cu[s] + (gb - p.blk_start[s]) * p.block;
  const int32_t q_off = p.offsets[h * nb + gb] + lo;
  for (int j = lane; j < nt; j += 32) {
    const int64_t left = rows - (int64_t)j * kTileRows;
    const int32_t nr = static_cast<int32_t>(left < kTileRows ? left : kTileRows);
    p.tdesc[t0 + j] = TileDesc{q_off, j * kTileRows, key0, h | (nr << 16)};
    p.tseg[t0 + j] = h * nb + gb;
  }
}

// grid (n_idx_tiles, h_k), block kIdxThreads; dynamic smem, in 32-bit words:
//   masks [idx_tok / 32][nb_max]: bit (t % 32) of word [t / 32][gb] is set when tile
//                                 token t kept block gb;
//   qbase, pbase [nb_max]:        the block's first q_list position and first
//                                 forward partial row for this tile's tokens;
//   wpre [idx_tok / 32][nb_max]:  bytes, tokens of earlier warps that kept gb.
size_t index_scatter_smem(const Params &p) {
  const size_t mw = p.idx_tok / 32;
  return 4 * (mw * p.nb_max + 2 * p.nb_max) + mw * p.nb_max + 16;
}

template <int TP>
__global__ void __launch_bounds__(kIdxThreads) scatter_kernel(Params p) {
  extern __shared__ uint32_t masks[];
  const int nb = *p.nb;
  const int h = blockIdx.y, tile = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const int mw = p.idx_tok >> 5;
  int32_t *qbase = reinterpret_cast<int32_t *>(masks + mw * p.nb_max);
  int32_t *pbase = qbase + p.nb_max;
  uint8_t *wpre = reinterpret_cast<uint8_t *>(pbase + p.nb_max);
  const int w = tile / p.wave_tiles;
  const int64_t hist_row = ((int64_t)h * p.n_idx_tiles + tile) * p.nb_max;
  const int64_t lo_row = ((int64_t)h * p.n_idx_tiles + (int64_t)w * p.wave_tiles) * p.nb_max;
  const int64_t sub_row = ((int64_t)h * p.n_w + w) * p.nb_max;
  {
    // mw * nb words from a 16-byte aligned start: four at a time, then the tail
    uint4 *m4 = reinterpret_cast<uint4 *>(masks);
    const int nw = mw * nb, n4 = nw >> 2;
    for (int i = tid; i < n4; i += blockDim.x) m4[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = 4 * n4 + tid; i < nw; i += blockDim.x) masks[i] = 0u;
  }
  for (int gb = tid; gb < nb; gb += blockDim.x) {
    const int32_t before = p.chunk_hist[hist_row + gb];   // earlier tokens of the block's list
    qbase[gb] = p.offsets[h * nb + gb] + before;
    pbase[gb] = p.wtile_off[sub_row + gb] * kTileRows + (before - p.chunk_hist[lo_row + gb]) * p.g;
  }
  __syncthreads();
  const int t0 = tile * p.idx_tok;
  const int t = t0 + tid;
  const bool live = tid < p.idx_tok && t < p.n;
  int32_t kgb[TP];
#pragma unroll
  for (int k = 0; k < TP; ++k) kgb[k] = -1;
  if (live && nb > 0) {
    bool bad = false;   // raised by the count pass already
    token_blocks<TP>(p, nb, h, t, kgb, bad);
  }
  {
    const bool on = live && nb > 0;
    const uint32_t act = __ballot_sync(0xffffffffu, on);
    if (on) {
      const int leader = __ffs(act) - 1;
      uint32_t *mrow = masks + (tid >> 5) * nb;
#pragma unroll
      for (int k = 0; k < TP; ++k) {
        const int32_t lead_gb = __shfl_sync(act, kgb[k], leader);
        const uint32_t same = __ballot_sync(act, kgb[k] == lead_gb && kgb[k] >= 0);
        if (kgb[k] >= 0) {
          if (kgb[k] != lead_gb) atomicOr(&mrow[kgb[k]], 1u << lane);
          else if (lane == leader) atomicOr(&mrow[kgb[k]], same);
        }
      }
    }
  }
  __syncthreads();
  // tokens of earlier warps per (warp, block)
  for (int gb = tid; gb < nb; gb += blockDim.x) {
    int run = 0;
    for (int w2 = 0; w2 < mw; ++w2) {
      wpre[w2 * nb + gb] = static_cast<uint8_t>(run);
      run += __popc(masks[w2 * nb + gb]);
    }
  }
  __syncthreads();
  if (live) {
    // this token's row of slot_map and prow, computed in registers and written with
    // 16-byte stores (the rows of a warp's tokens are contiguous)
    const int wl = tid >> 5;
    const uint32_t below = (1u << lane) - 1u;
    int32_t srow[TP], prw[TP];
#pragma unroll
    for (int k = 0; k < TP; ++k) {
      const int gb = kgb[k];
      srow[k] = -1;
      prw[k] = -1;
      if (k < p.topk && gb >= 0) {
        const int32_t r = __popc(masks[wl * nb + gb] & below) + wpre[wl * nb + gb];
        const int32_t pos = qbase[gb] + r;
        p.q_list[pos] = t;
        srow[k] = pos;
        prw[k] = pbase[gb] + r * p.g;
      }
    }
    const int64_t base = ((int64_t)h * p.n + t) * p.topk;
    if (TP == p.topk && (TP % 4) == 0) {
      int4 *ds = reinterpret_cast<int4 *>(p.slot_map + base);
      int4 *dp = reinterpret_cast<int4 *>(p.prow + base);
#pragma unroll
      for (int k = 0; k < TP; k += 4) {
        ds[k / 4] = make_int4(srow[k], srow[k + 1], srow[k + 2], srow[k + 3]);
        dp[k / 4] = make_int4(prw[k], prw[k + 1], prw[k + 2], prw[k + 3]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < TP; ++k) {
        if (k < p.topk) {
          p.slot_map[base + k] = srow[k];
          p.prow[base + k] = prw[k];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Host launcher
// ---------------------------------------------------------------------------
template <int TP>
static void launch_count_scatter(const Params &p, bool scatter, dim3 grid, size_t smem,
                                 cudaStream_t stream) {
  if (scatter)
    scatter_kernel<TP><<<grid, kIdxThreads, smem, stream>>>(p);
  else
    count_kernel<TP><<<grid, kIdxThreads, smem, stream>>>(p);
}

static void count_or_scatter(const Params &p, bool scatter, dim3 grid, size_t smem,
                             cudaStream_t s) {
  if (p.topk <= 1) launch_count_scatter<1>(p, scatter, grid, smem, s);
  else if (p.topk <= 2) launch_count_scatter<2>(p, scatter, grid, smem, s);
  else if (p.topk <= 4) launch_count_scatter<4>(p, scatter, grid, smem, s);
  else if (p.topk <= 8) launch_count_scatter<8>(p, scatter, grid, smem, s);
  else if (p.topk <= 16) launch_count_scatter<16>(p, scatter, grid, smem, s);
  else launch_count_scatter<32>(p, scatter, grid, smem, s);
}

size_t index_count_smem(const Params &p) { return sizeof(int32_t) * p.nb_max; }
size_t index_scatter_smem(const Params &p);

cudaError_t launch_index(const Params &p, cudaStream_t stream, void (*mark)(int, cudaStream_t, bool)) {
  mark(0, stream, true);
  geometry_kernel<<<1, 1024, 0, stream>>>(p);
  mark(0, stream, false);
  const dim3 grid_t(static_cast<unsigned>(p.n_idx_tiles), p.h_k);
  mark(1, stream, true);
  count_or_scatter(p, false, grid_t, index_count_smem(p), stream);
  mark(1, stream, false);
  mark(2, stream, true);
  col_scan_kernel<<<dim3(static_cast<unsigned>((p.nb_max + 31) / 32), p.h_k), dim3(32, 32), 0,
                    stream>>>(p);
  mark(2, stream, false);
  mark(3, stream, true);
  scan_kernel<<<1, 1024, 0, stream>>>(p);
  if (p.n_w > 1) {   // with one wave scan_kernel has written wtile_off already
    wave_scan_local_kernel<<<static_cast<unsigned>(p.n_scan_ctas), 1024, 0, stream>>>(p);
    wave_scan_add_kernel<<<static_cast<unsigned>(p.n_scan_ctas), 1024, 0, stream>>>(p);
  }
  tile_desc_kernel<<<static_cast<unsigned>((p.nsub + 7) / 8), 256, 0, stream>>>(p);
  mark(3, stream, false);
  mark(4, stream, true);
  count_or_scatter(p, true, grid_t, index_scatter_smem(p), stream);
  mark(4, stream, false);
  return cudaGetLastError();
}

template <int TP>
static cudaError_t set_limits_tp(int count_smem, int scatter_smem) {
  cudaError_t e = cudaFuncSetAttribute(count_kernel<TP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, count_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(scatter_kernel<TP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              scatter_smem);
}

cudaError_t index_set_smem_limits(const Params &p) {
  const int cs = static_cast<int>(index_count_smem(p)), ss = static_cast<int>(index_scatter_smem(p));
  if (p.topk <= 1) return set_limits_tp<1>(cs, ss);
  if (p.topk <= 2) return set_limits_tp<2>(cs, ss);
  if (p.topk <= 4) return set_limits_tp<4>(cs, ss);
  if (p.topk <= 8) return set_limits_tp<8>(cs, ss);
  if (p.topk <= 16) return set_limits_tp<16>(cs, ss);
  return set_limits_tp<32>(cs, ss);
}

}  // namespace nsa
