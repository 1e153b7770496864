// compress.cu -- the step before selected attention: compression of keys and values,
// attention over the compressed tokens, block importance and top-T block selection,
// producing the selection rows the selected-attention kernels take (Native Sparse
// Attention's compression and selection branches, papernotes page, 领域现状 and the
// 方法详解 flowchart's "NSA 稀疏选择张量 T"; hyperparameters of the
// Flash-Sparse-Attention README's "Usage": kernel_size 32, kernel_stride 16,
// block_size 64, topk 16, init_blocks 1, local_blocks 2).
//
// The pages give no compression formula: compressed token i of a sequence is the
// mean of its keys (values) at positions [i*stride, i*stride + l); the query at
// position tau sees it when i*stride + l - 1 <= tau.  The importance of selection
// block j is the summed probability, over the group's g query heads, of the visible
// compressed tokens whose window overlaps the block's keys.  Top-T keeps the init
// and local blocks first (ascending), then the others by importance, ties to the
// lower block.
//
// cmp_attn_select_kernel: one CTA per (KV head, TT consecutive tokens); rows are
// (token, query head of the group) pairs, 16 per warp, on mma.sync m16n8k16 with
// fp32 accumulators.  Pass 1 is an online-softmax attention over 64-token chunks of
// compressed keys (out, lse); pass 2 recomputes the scores, forms the exact
// probabilities from lse and adds them into a shared-memory importance row per
// token; a warp per token then takes the top T.
#include "compress.cuh"

namespace nsa {

// Offsets of each sequence's compressed tokens (one CTA, 1024 threads); also checks
// cu_seqlens (starts at 0, non-decreasing, ends at n).
__global__ void __launch_bounds__(1024) cmp_offsets_kernel(const int32_t *cu, int num_seqs, int n,
                                                           int ksize, int stride, int32_t *cu_cmp,
                                                           int32_t *status) {
  __shared__ int32_t part[1024];
  const int tid = threadIdx.x;
  const int per = (num_seqs + 1023) / 1024;
  const int s0 = min(num_seqs, tid * per), s1 = min(num_seqs, s0 + per);
  int32_t sum = 0;
  bool bad = false;
  for (int s = s0; s < s1; ++s) {
    const int len = cu[s + 1] - cu[s];
    bad |= len < 0;
    sum += len >= ksize ? (len - ksize) / stride + 1 : 0;
  }
  part[tid] = sum;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {   // inclusive scan
    const int32_t x = tid >= off ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += x;
    __syncthreads();
  }
  int32_t run = tid ? part[tid - 1] : 0;
  for (int s = s0; s < s1; ++s) {
    cu_cmp[s] = run;
    const int len = cu[s + 1] - cu[s];
    run += len >= ksize ? (len - ksize) / stride + 1 : 0;
  }
  if (tid == 1023) cu_cmp[num_seqs] = part[1023];
  if (tid == 0) bad |= cu[0] != 0 || cu[num_seqs] != n;
  if (__syncthreads_or(bad) && tid == 0 && status) set_status(status, NSA_DEVERR_BAD_SEQLENS);
}

// kc[r, h] = mean of k over compressed token r's window, likewise vc; one warp per
// (row, KV head), fp32 sums.
template <int D, bool kFp16>
__global__ void __launch_bounds__(256) compress_kernel(const int32_t *cu, const int32_t *cu_cmp,
                                                       int num_seqs, int n, int h_k, int ksize,
                                                       int stride, int64_t rows_cap,
                                                       const void *k, const void *v, void *kc,
                                                       void *vc) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (w >= rows_cap * h_k) return;
  const int r = static_cast<int>(w / h_k), h = static_cast<int>(w % h_k);
  if (r >= __ldg(cu_cmp + num_seqs)) return;
  const int s = seq_of(cu_cmp, num_seqs, r);
  const int64_t a = __ldg(cu + s) + (int64_t)(r - __ldg(cu_cmp + s)) * stride;
  if (a < 0 || a + ksize > n) return;   // malformed cu_seqlens (flagged by the offsets)
  float ak[E], av[E];
#pragma unroll
  for (int e = 0; e < E; ++e) ak[e] = av[e] = 0.f;
  const uint16_t *pk = static_cast<const uint16_t *>(k) + (a * h_k + h) * D + lane * E;
  const uint16_t *pv = static_cast<const uint16_t *>(v) + (a * h_k + h) * D + lane * E;
  for (int j = 0; j < ksize; ++j) {
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 x = unpack2<kFp16>(__ldg(reinterpret_cast<const uint32_t *>(pk + e)));
      const float2 y = unpack2<kFp16>(__ldg(reinterpret_cast<const uint32_t *>(pv + e)));
      ak[e] += x.x;
      ak[e + 1] += x.y;
      av[e] += y.x;
      av[e + 1] += y.y;
    }
    pk += (int64_t)h_k * D;
    pv += (int64_t)h_k * D;
  }
  const float inv = 1.f / static_cast<float>(ksize);
  uint16_t *ok = static_cast<uint16_t *>(kc) + ((int64_t)r * h_k + h) * D + lane * E;
  uint16_t *ov = static_cast<uint16_t *>(vc) + ((int64_t)r * h_k + h) * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    *reinterpret_cast<uint32_t *>(ok + e) = pack2<kFp16>(ak[e] * inv, ak[e + 1] * inv);
    *reinterpret_cast<uint32_t *>(ov + e) = pack2<kFp16>(av[e] * inv, av[e + 1] * inv);
  }
}

// ---------------------------------------------------------------------------
// mma.sync m16n8k16 (fp32 accumulate) and ldmatrix
// ---------------------------------------------------------------------------
template <bool kFp16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (kFp16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

constexpr int kCmpChunk = 64;   // compressed tokens per chunk
constexpr int kPsStride = 68;   // floats per row of the probability tile

template <int D>
struct CmpSmem {
  static constexpr int kRow = D + 8;                                // padded row (16-bit)
  static constexpr int kBuf = kCmpChunk * kRow * 2;                 // one K or V chunk
  static constexpr int kK = 0;                                      // K: 2 buffers
  static constexpr int kV = 2 * kBuf;                               // V: 2 buffers
  static constexpr int kPsMax = 128 * kPsStride * 4;                // pass-2 tile (aliases V)
  static constexpr int kImp = kV + (2 * kBuf > kPsMax ? 2 * kBuf : kPsMax);
  static size_t bytes(int tt, int nb_max) { return kImp + (size_t)tt * nb_max * 4; }
};

template <int D, bool kFp16>
__global__ void __launch_bounds__(256) cmp_attn_select_kernel(const CmpParams p) {
  using L = CmpSmem<D>;
  constexpr int KS = D / 16;        // k-steps of the score MMA
  constexpr int NT = kCmpChunk / 8; // score n-tiles per chunk
  extern __shared__ __align__(128) uint8_t smem[];
  // importance rows: this CTA's slice of the caller's workspace when given, else
  // shared memory
  float *imp = p.imp_ws ? p.imp_ws + ((int64_t)blockIdx.y * gridDim.x + blockIdx.x) *
                                         p.tt * p.nb_max
                        : reinterpret_cast<float *>(smem + L::kImp);
  float *ps = reinterpret_cast<float *>(smem + L::kV);
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int grp = lane >> 2, qd = lane & 3;
  const int hk = blockIdx.y;
  const int t0 = blockIdx.x * p.tt;
  if (t0 >= p.n) return;
  const int t_end = min(t0 + p.tt, p.n);
  const int rows = p.tt * p.g;
  const uint16_t *kc = static_cast<const uint16_t *>(p.kc);
  const uint16_t *vc = static_cast<const uint16_t *>(p.vc);
  const uint64_t keep = l2_evict_last();
  const bool quad = p.block == 4 * p.stride && p.ksize == 2 * p.stride;

  const int s_first = seq_of(p.cu, p.num_seqs, t0);
  const int s_last = seq_of(p.cu, p.num_seqs, t_end - 1);
  for (int s = s_first; s <= s_last; ++s) {
    const int cs = __ldg(p.cu + s), ce = __ldg(p.cu + s + 1);
    const int a = max(t0, cs), b = min(t_end, ce);
    if (a >= b) continue;
    const int cbase = __ldg(p.cu_cmp + s);
    const int taub = b - 1 - cs;   // the last token's position
    const int nv_max = taub >= p.ksize - 1 ? (taub - p.ksize + 1) / p.stride + 1 : 0;
    // malformed offsets or a sequence longer than max_seqlen: flag, skip its tokens
    if (cs < 0 || ce > p.n || ce - cs > p.max_seqlen || cbase < 0 ||
        (int64_t)cbase + nv_max > p.rows_cap) {
      if (tid == 0 && p.status) set_status(p.status, NSA_DEVERR_BAD_SEQLENS);
      continue;
    }
    const int nchunks = (nv_max + kCmpChunk - 1) / kCmpChunk;

    // this thread's two rows: r0 = warp*16 + grp, r1 = r0 + 8
    int nv[2], tok[2], hq[2];
    bool act[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = warp * 16 + grp + u * 8;
      tok[u] = t0 + r / p.g;
      hq[u] = hk * p.g + r % p.g;
      act[u] = r < rows && tok[u] >= a && tok[u] < b;
      const int tau = tok[u] - cs;
      nv[u] = act[u] && tau >= p.ksize - 1 ? (tau - p.ksize + 1) / p.stride + 1 : 0;
    }
    // Q fragments (A operand), zeros for inactive rows
    uint32_t qa[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t *qr = reinterpret_cast<const uint32_t *>(
            static_cast<const uint16_t *>(p.q) + ((int64_t)tok[u] * p.h_q + hq[u]) * D);
        qa[ks][u] = act[u] ? __ldg(qr + ks * 8 + qd) : 0u;
        qa[ks][u + 2] = act[u] ? __ldg(qr + ks * 8 + 4 + qd) : 0u;
      }
    }

    // Chunk c's compressed rows into buffer c & 1 (rows past nv_max repeat the last
    // visible row: finite values whose probabilities are masked to 0).
    auto load_chunk = [&](int c, bool with_v) {
      const int per_row = D / 8;
      const int total = kCmpChunk * per_row;
      for (int i = tid; i < total; i += blockDim.x) {
        const int r = i / per_row, ch = i % per_row;
        const int row = cbase + min(c * kCmpChunk + r, nv_max - 1);
        const int64_t goff = ((int64_t)row * p.h_k + hk) * D + ch * 8;
        const uint32_t soff = (c & 1) * L::kBuf + (r * L::kRow + ch * 8) * 2;
        cp_async16_hint(sbase + L::kK + soff, kc + goff, 16, keep);
        if (with_v) cp_async16_hint(sbase + L::kV + soff, vc + goff, 16, keep);
      }
      cp_async_commit();
    };
    // S = Q Kc^T for chunk c: sc[nt][0..1] row r0 cols 8nt + 2qd (+1), [2..3] row r1
    auto scores = [&](int c, float (&sc)[NT][4]) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      const uint32_t kb = sbase + L::kK + (c & 1) * L::kBuf;
      const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int key = np * 16 + (mi >> 1) * 8 + ri, dim = ks * 16 + (mi & 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + (key * L::kRow + dim) * 2, b0, b1, b2, b3);
          mma16816<kFp16>(sc[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
          mma16816<kFp16>(sc[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
      }
    };

    // ---------------- pass 1: out and lse ----------------
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[D / 8][4];
#pragma unroll
    for (int j = 0; j < D / 8; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    if (nchunks > 0) load_chunk(0, true);
    for (int c = 0; c < nchunks; ++c) {
      if (c + 1 < nchunks) {
        load_chunk(c + 1, true);
        cp_async_wait_group<1>();
      } else {
        cp_async_wait_group<0>();
      }
      __syncthreads();
      float sc[NT][4];
      scores(c, sc);
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = c * kCmpChunk + nt * 8 + 2 * qd + (e & 1);
          if (col >= nv[e >> 1]) sc[nt][e] = -INFINITY;
          mx[e >> 1] = fmaxf(mx[e >> 1], sc[nt][e]);
        }
      float alpha[2], mu[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        mx[u] = fmaxf(mx[u], __shfl_xor_sync(0xffffffffu, mx[u], 1));
        mx[u] = fmaxf(mx[u], __shfl_xor_sync(0xffffffffu, mx[u], 2));
        const float mn = fmaxf(m[u], mx[u]);
        mu[u] = mn == -INFINITY ? 0.f : mn * p.scale_log2;
        alpha[u] = ex2_approx(m[u] * p.scale_log2 - mu[u]);   // 0 while m = -inf
        m[u] = mn;
        l[u] *= alpha[u];
      }
#pragma unroll
      for (int j = 0; j < D / 8; ++j) {
        o[j][0] *= alpha[0];
        o[j][1] *= alpha[0];
        o[j][2] *= alpha[1];
        o[j][3] *= alpha[1];
      }
      uint32_t pa[NT][2];   // P rounded to 16 bits, packed as A fragments
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pv[e] = ex2_approx(fmaf(sc[nt][e], p.scale_log2, -mu[e >> 1]));   // -inf -> 0
          l[e >> 1] += pv[e];
        }
        pa[nt][0] = pack2<kFp16>(pv[0], pv[1]);
        pa[nt][1] = pack2<kFp16>(pv[2], pv[3]);
      }
      // O += P V
      const uint32_t vb = sbase + L::kV + (c & 1) * L::kBuf;
      const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
      for (int kk = 0; kk < NT / 2; ++kk) {
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int key = kk * 16 + (mi & 1) * 8 + ri, dim = dp * 16 + (mi >> 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + (key * L::kRow + dim) * 2, b0, b1, b2, b3);
          mma16816<kFp16>(o[2 * dp], pa[2 * kk][0], pa[2 * kk][1], pa[2 * kk + 1][0],
                          pa[2 * kk + 1][1], b0, b1);
          mma16816<kFp16>(o[2 * dp + 1], pa[2 * kk][0], pa[2 * kk][1], pa[2 * kk + 1][0],
                          pa[2 * kk + 1][1], b2, b3);
        }
      }
      __syncthreads();
    }
    float lse2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      l[u] += __shfl_xor_sync(0xffffffffu, l[u], 1);
      l[u] += __shfl_xor_sync(0xffffffffu, l[u], 2);
      lse2[u] = l[u] > 0.f ? m[u] * p.scale_log2 + __log2f(l[u]) : -INFINITY;
      const float inv = l[u] > 0.f ? 1.f / l[u] : 0.f;
      if (act[u]) {
        uint32_t *orow = reinterpret_cast<uint32_t *>(
            static_cast<uint16_t *>(p.out) + ((int64_t)tok[u] * p.h_q + hq[u]) * D);
#pragma unroll
        for (int j = 0; j < D / 8; ++j)
          orow[j * 4 + qd] = pack2<kFp16>(o[j][2 * u] * inv, o[j][2 * u + 1] * inv);
        if (qd == 0) p.lse[(int64_t)hq[u] * p.n + tok[u]] = lse2[u] * 0.69314718055994531f;
      }
    }

    // ---------------- pass 2: block importance ----------------
    const int tl0 = a - t0, ntok = b - a;
    const int nb_cta = taub / p.block + 1;
    for (int i = tid; i < ntok * nb_cta; i += blockDim.x)
      imp[(tl0 + i / nb_cta) * p.nb_max + i % nb_cta] = 0.f;
    __syncthreads();
    if (nchunks > 0) load_chunk(0, false);
    for (int c = 0; c < nchunks; ++c) {
      if (c + 1 < nchunks) {
        load_chunk(c + 1, false);
        cp_async_wait_group<1>();
      } else {
        cp_async_wait_group<0>();
      }
      __syncthreads();
      float sc[NT][4];
      scores(c, sc);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = c * kCmpChunk + nt * 8 + 2 * qd + (e & 1);
          pv[e] = col < nv[e >> 1] ? ex2_approx(fmaf(sc[nt][e], p.scale_log2, -lse2[e >> 1]))
                                   : 0.f;
        }
        const int r0 = warp * 16 + grp;
        *reinterpret_cast<float2 *>(ps + r0 * kPsStride + nt * 8 + 2 * qd) =
            make_float2(pv[0], pv[1]);
        *reinterpret_cast<float2 *>(ps + (r0 + 8) * kPsStride + nt * 8 + 2 * qd) =
            make_float2(pv[2], pv[3]);
      }
      __syncthreads();
      // (token, block) pairs this chunk touches; each is owned by one thread
      const int i0 = c * kCmpChunk, i1 = min(i0 + kCmpChunk, nv_max) - 1;
      const int j0 = i0 * p.stride / p.block;
      const int j1 = (i1 * p.stride + p.ksize - 1) / p.block;
      const int nj = j1 - j0 + 1;
      for (int w = tid; w < ntok * nj; w += blockDim.x) {
        const int tl = tl0 + w / nj, j = j0 + w % nj;
        float acc = 0.f;
        if (quad) {
          // B = 4 stride, l = 2 stride: block j - j0 is overlapped by the chunk's
          // windows 4 (j - j0) - 1 .. 4 (j - j0) + 3 (columns past the visible ones
          // hold 0); the first of them belongs to the previous chunk when j = j0
          const int jr = j - j0;
          for (int h = 0; h < p.g; ++h) {
            const float *prow = ps + (tl * p.g + h) * kPsStride;
            if (jr < kCmpChunk / 4) {
              const float4 x = *reinterpret_cast<const float4 *>(prow + 4 * jr);
              acc += (x.x + x.y) + (x.z + x.w);
            }
            if (jr >= 1) acc += prow[4 * jr - 1];
          }
        } else {
          // windows overlapping keys [j*B, j*B + B): i*stride < j*B + B, i*stride + l > j*B
          const int lo_num = j * p.block - p.ksize + 1;
          const int ilo = max(i0, lo_num > 0 ? (lo_num + p.stride - 1) / p.stride : 0);
          const int ihi = min(i1, (j * p.block + p.block - 1) / p.stride);
          for (int h = 0; h < p.g; ++h) {
            const float *prow = ps + (tl * p.g + h) * kPsStride - i0;
            for (int i = ilo; i <= ihi; ++i) acc += prow[i];
          }
        }
        imp[tl * p.nb_max + j] += acc;
      }
      __syncthreads();
    }

    // ---------------- top-T per token ----------------
    for (int tl = tl0 + warp; tl < tl0 + ntok; tl += nwarps) {
      const int t = t0 + tl, tau = t - cs, cblk = tau / p.block;
      float *row = imp + tl * p.nb_max;
      int32_t *out_sel = p.sel + ((int64_t)hk * p.n + t) * p.topk;
      for (int k = 0; k < p.topk; ++k) {
        float bv = -1.f;
        int bj = 0x7fffffff;
        for (int j = lane; j <= cblk; j += 32) {
          const float x = row[j];
          if (x < 0.f) continue;   // taken
          const float v = (j < p.init_blocks || j > cblk - p.local_blocks) ? INFINITY : x;
          if (v > bv) { bv = v; bj = j; }   // ascending j per lane: ties keep the lower
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
          const int oj = __shfl_xor_sync(0xffffffffu, bj, off);
          if (ov > bv || (ov == bv && oj < bj)) { bv = ov; bj = oj; }
        }
        if (lane == 0) out_sel[k] = bj == 0x7fffffff ? -1 : bj;
        if (bj != 0x7fffffff && lane == (bj & 31)) row[bj] = -1.f;
        __syncwarp();
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_cmp_offsets(const int32_t *cu, int num_seqs, int n, int ksize, int stride,
                               int32_t *cu_cmp, int32_t *status, cudaStream_t s) {
  cmp_offsets_kernel<<<1, 1024, 0, s>>>(cu, num_seqs, n, ksize, stride, cu_cmp, status);
  return cudaGetLastError();
}

template <int D, bool kFp16>
static cudaError_t run_compress(const int32_t *cu, const int32_t *cu_cmp, int num_seqs, int n,
                                int h_k,
                                int ksize, int stride, int64_t rows_cap, const void *k,
                                const void *v, void *kc, void *vc, cudaStream_t s) {
  const int64_t warps = rows_cap * h_k;
  if (warps <= 0) return cudaSuccess;
  compress_kernel<D, kFp16><<<static_cast<unsigned>((warps + 7) / 8), 256, 0, s>>>(
      cu, cu_cmp, num_seqs, n, h_k, ksize, stride, rows_cap, k, v, kc, vc);
  return cudaGetLastError();
}

cudaError_t launch_compress(int d, bool fp16, const int32_t *cu, const int32_t *cu_cmp,
                            int num_seqs, int n, int h_k, int ksize, int stride,
                            int64_t rows_cap,
                            const void *k, const void *v, void *kc, void *vc, cudaStream_t s) {
  switch (d) {
    case 64:
      return fp16 ? run_compress<64, true>(cu, cu_cmp, num_seqs, n, h_k, ksize, stride, rows_cap, k,
                                           v, kc, vc, s)
                  : run_compress<64, false>(cu, cu_cmp, num_seqs, n, h_k, ksize, stride, rows_cap,
                                            k, v, kc, vc, s);
    case 128:
      return fp16 ? run_compress<128, true>(cu, cu_cmp, num_seqs, n, h_k, ksize, stride, rows_cap,
                                            k, v, kc, vc, s)
                  : run_compress<128, false>(cu, cu_cmp, num_seqs, n, h_k, ksize, stride, rows_cap,
                                             k, v, kc, vc, s);
    default: return cudaErrorInvalidValue;
  }
}

// Tokens per CTA: the largest power of two <= 128 with at most 128 rows (8 warps) and,
// when the importance rows live in shared memory (in_smem), those rows within it;
// 0 when none fits.
int cmp_tokens_per_cta(int d, int g, int nb_max, bool in_smem) {
  const size_t limit = 227 * 1024;
  for (int tt = 128; tt >= 1; tt >>= 1) {
    if (tt * g > 128) continue;
    if (!in_smem) return tt;
    const size_t bytes = d == 64 ? CmpSmem<64>::bytes(tt, nb_max) : CmpSmem<128>::bytes(tt, nb_max);
    if (bytes <= limit) return tt;
  }
  return 0;
}

template <int D, bool kFp16>
static cudaError_t run_cmp_select(const CmpParams &p, cudaStream_t s) {
  const size_t smem = p.imp_ws ? CmpSmem<D>::kImp : CmpSmem<D>::bytes(p.tt, p.nb_max);
  auto kern = cmp_attn_select_kernel<D, kFp16>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int warps = (p.tt * p.g + 15) / 16;
  dim3 grid((p.n + p.tt - 1) / p.tt, p.h_k);
  kern<<<grid, warps * 32, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_cmp_select(int d, bool fp16, const CmpParams &p, cudaStream_t s) {
  if (p.n <= 0) return cudaSuccess;
  switch (d) {
    case 64: return fp16 ? run_cmp_select<64, true>(p, s) : run_cmp_select<64, false>(p, s);
    case 128: return fp16 ? run_cmp_select<128, true>(p, s) : run_cmp_select<128, false>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nsa
