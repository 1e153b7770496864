// bwd.cu -- backward of NSA selected attention on sm_103a.
//
// Same KV-block-outer order and the same tiles as the forward ("FSA: An
// Alternative Efficient Implementation of Native Sparse Attention Kernel", key
// designs 1-2; the backward reuses the forward's index tensors I_i / O_i):
//
//   bwd_pre   : D[hq, t] = sum_d dO * O (fp32); the first dK/dV partial slot of
//               every (KV head, block) segment.
//   bwd_main  : persistent and warp-specialised; tiles are dealt to the CTAs in
//               chunks of consecutive tiles.  Per tile, on tcgen05 with TMEM
//               accumulators: S = Q K_b^T and dP = dO V_b^T; in registers P =
//               exp2(S*scale*log2e - lse*log2e) (causal mask) and dS = P (dP - D),
//               written to shared memory in 16 bits; dV_b^T += dO^T P and dK_b^T +=
//               Q^T dS stay in TMEM over a run of tiles of one block inside one
//               chunk; dQ_part = dS K_b goes to a tile-padded compact buffer.  At the
//               end of a run the dK_b, dV_b partials are written once (one slot per
//               block and chunk).
//   bwd_dq    : per (token, query head), dq = scale * sum of its <= T dQ partials.
//   bwd_dkv   : per block, dk = scale * sum of its partials of dK, dv = that of dV;
//               blocks nobody selected get zeros.
// No atomics decide any sum, so the result is bit-reproducible.
#include "common.cuh"

namespace nsa {

// ---------------------------------------------------------------------------
// D = rowsum(dO * O): one warp per four (token, query head) rows
// ---------------------------------------------------------------------------
template <int D, bool kFp16>
__global__ void __launch_bounds__(256) bwd_pre_kernel(Params p) {
  // four rows per warp, their loads issued together
  constexpr int E = D / 32, R = 4;
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)p.n * p.h_q;
  const int64_t r0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * R;
  if (r0 >= rows) return;
  uint32_t a[R][E / 2], b[R][E / 2];
#pragma unroll
  for (int k = 0; k < R; ++k) {
    const int64_t r = min(r0 + k, rows - 1);
    const uint16_t *o = static_cast<const uint16_t *>(p.out_in) + r * D + lane * E;
    const uint16_t *g = static_cast<const uint16_t *>(p.dout) + r * D + lane * E;
    if constexpr (E == 2) {
      a[k][0] = __ldcs(reinterpret_cast<const unsigned int *>(o));
      b[k][0] = __ldcs(reinterpret_cast<const unsigned int *>(g));
    } else if constexpr (E == 4) {
      const uint2 x = __ldcs(reinterpret_cast<const uint2 *>(o));
      const uint2 y = __ldcs(reinterpret_cast<const uint2 *>(g));
      a[k][0] = x.x; a[k][1] = x.y; b[k][0] = y.x; b[k][1] = y.y;
    } else {
      const uint4 x = __ldcs(reinterpret_cast<const uint4 *>(o));
      const uint4 y = __ldcs(reinterpret_cast<const uint4 *>(g));
      a[k][0] = x.x; a[k][1] = x.y; a[k][2] = x.z; a[k][3] = x.w;
      b[k][0] = y.x; b[k][1] = y.y; b[k][2] = y.z; b[k][3] = y.w;
    }
  }
#pragma unroll
  for (int k = 0; k < R; ++k) {
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < E / 2; ++e) {
      const float2 x = unpack2<kFp16>(a[k][e]);
      const float2 y = unpack2<kFp16>(b[k][e]);
      acc = fmaf(x.x, y.x, fmaf(x.y, y.y, acc));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    const int64_t r = r0 + k;
    if (lane == 0 && r < rows) {
      const int t = static_cast<int>(r / p.h_q), hq = static_cast<int>(r - (int64_t)t * p.h_q);
      p.dstat[(int64_t)hq * p.n + t] = acc;
    }
  }
}

// First dK/dV partial slot of every segment.  The main kernel deals tiles in
// chunks of C = p.bwd_chunk consecutive tiles and writes one dK/dV partial per
// (segment, chunk) pair the segment's tiles meet, so a segment with tiles
// [a, b) gets (b - 1) / C - a / C + 1 slots.  One block of 1024 threads.
__global__ void __launch_bounds__(1024) bwd_parts_kernel(Params p) {
  __shared__ int32_t sums[32];
  const int nseg = p.h_k * (*p.nb);
  const int per = p.bwd_chunk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int each = (nseg + 1023) / 1024;
  const int i0 = min(nseg, tid * each), i1 = min(nseg, i0 + each);
  auto parts = [&](int i) {
    const int a = p.tile_off[i], b = p.tile_off[i + 1];
    return b > a ? (b - 1) / per - a / per + 1 : 0;
  };
  int32_t local = 0;
  for (int i = i0; i < i1; ++i) local += parts(i);
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
  for (int i = i0; i < i1; ++i) {
    p.part_off[i] = run;
    run += parts(i);
  }
  if (tid == 1023) p.part_off[nseg] = sums[31];
}

// ---------------------------------------------------------------------------
// Main kernel configuration per (d, B_K)
// ---------------------------------------------------------------------------
template <int D, int BK>
struct BwdCfg {
  static constexpr int DW = D < 128 ? 128 : D;   // Q / dO tile width (d = 64 padded with zeros)
  static constexpr int NH = D == 256 ? 2 : 1;    // 128-row halves of dK^T, dV^T; dQ column halves
  static constexpr int DQC = D < 128 ? D : 128;  // dQ columns per half
  static constexpr int NKV = BK < 64 ? 64 : BK;  // P / dS columns: at least one 128-byte atom
  static constexpr int QS = (D == 256 || (D == 128 && BK == 128)) ? 1 : 2;   // Q/dO stages
  // compute warpgroups, each with its own S/dP (TMEM) and P/dS (shared memory)
  // buffers and taking every NWG-th tile; two where TMEM and shared memory have room
  static constexpr int NWG = (D <= 128 && BK <= 64) ? 2 : 1;
  static constexpr int NPW = 4;                  // producer warps
  static constexpr int WPS = NPW / QS;           // producer warps per Q/dO stage
  static constexpr int RW = 128 / WPS;           // tile rows gathered per producer warp
  // warps 0-3 producers, 4 MMA, 5 TMEM, 6 K/V, 8-11 (and 12-15) compute warpgroups
  static constexpr int kThreads = 256 + 128 * NWG;
  static constexpr uint32_t kQ = 128u * DW * 2u;        // one Q (or dO) tile
  static constexpr uint32_t kK = uint32_t(BK) * D * 2u;  // K or V
  static constexpr uint32_t kP = 128u * NKV * 2u;       // P or dS (also dQ staging)
  static constexpr uint32_t kOffQ = 0;                   // stage s: Q at 2 s kQ, dO at (2 s + 1) kQ
  static constexpr uint32_t kOffK = QS * 2 * kQ;
  static constexpr uint32_t kOffV = kOffK + kK;
  static constexpr uint32_t kOffP = kOffV + kK;          // warpgroup w: P at 2 w kP, dS after it
  static constexpr uint32_t kBytes = kOffP + NWG * 2 * kP + 1024;
  static_assert(kBytes <= 227u * 1024u, "shared memory budget");
  static_assert(2 * kP >= 128u * DQC * 2u, "P/dS buffers double as dQ staging");
  // TMEM: warpgroup w's S at [2 w BK, 2 w BK + BK) and dP at [2 w BK + BK, 2 (w + 1) BK);
  // dQ after them, or over them when short of columns (one warpgroup only); dV^T then
  // dK^T (NH lane halves of NKV columns each)
  static constexpr bool kDqAlias = NWG * 2 * BK + DQC + 2 * NH * NKV > 512;
  static_assert(!kDqAlias || NWG == 1, "an aliased dQ needs a single warpgroup");
  static constexpr int kTmDQ = kDqAlias ? 0 : NWG * 2 * BK;
  static constexpr int kTmDV = kDqAlias ? 2 * BK : NWG * 2 * BK + DQC;
  static constexpr int kTmDK = kTmDV + NH * NKV;
  static_assert(kTmDK + NH * NKV <= 512, "TMEM budget");
  static_assert(!kDqAlias || DQC <= 2 * BK, "aliased dQ fits the S/dP columns");
};

// 32 values of a row, already packed in 16-bit pairs, into four 16-byte chunks of a
// 128-byte-swizzled operand tile
__device__ __forceinline__ void st_row_packed(uint32_t tile, int row, int chunk0, const uint32_t *pk) {
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint32_t so = sw128_offset(row, chunk0 + q4, 128);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tile + so), "r"(pk[q4 * 4]),
                 "r"(pk[q4 * 4 + 1]), "r"(pk[q4 * 4 + 2]), "r"(pk[q4 * 4 + 3])
                 : "memory");
  }
}

template <bool kFp16>
__device__ __forceinline__ void st_row_chunks(uint32_t tile, int row, int chunk0, const float *v32) {
  uint32_t pk[16];
#pragma unroll
  for (int j = 0; j < 32; j += 2) pk[j / 2] = pack2<kFp16>(v32[j], v32[j + 1]);
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) {
    const uint32_t so = sw128_offset(row, chunk0 + q4, 128);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tile + so), "r"(pk[q4 * 4]),
                 "r"(pk[q4 * 4 + 1]), "r"(pk[q4 * 4 + 2]), "r"(pk[q4 * 4 + 3])
                 : "memory");
  }
}

// Persistent, warp-specialised backward main kernel (one CTA per SM).  Tiles are
// dealt to the CTAs in chunks of p.bwd_chunk consecutive tiles, round-robin, so all
// CTAs work on neighbouring blocks at any time and the Q/dO rows they gather stay
// L2-resident.  A run is a CTA's consecutive tiles of one (KV head, block) inside one
// chunk: K/V is loaded, and dK/dV accumulated in TMEM, once per run.
//   warps 0-3: producers -- the WPS warps of a Q/dO stage gather RW rows each of
//     that stage's tiles by cp.async into the 128-byte-swizzled operand layout and
//     arrive when their own copies have landed;
//   warp 6 (one thread): K_b and V_b by TMA, once per run;
//   warp 4 (one thread): tcgen05 MMAs, per tile S and dP (interleaved: two
//     independent accumulators), then dV^T, dK^T and dQ.  S/dP of later tiles are
//     issued as soon as their Q/dO rows have landed, while it waits for P/dS;
//   warps 8-11 (and 12-15): compute warpgroup w takes tiles w, w + NWG, ...: P and
//     dS of its tile, the dQ epilogue (through its P/dS buffers, free once the dQ
//     MMA has read them) and, at the end of a run, dK/dV out.
// mbarriers hand each buffer between roles; every wait is bounded.
// kWin: the sliding window's lower key bound is applied (p.window > 0).
template <int D, int BK, bool kFp16, bool kWin>
__global__ void __launch_bounds__(BwdCfg<D, BK>::kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_dq, Params p) {
  using L = BwdCfg<D, BK>;
  constexpr int QS = L::QS, NWG = L::NWG, NH = L::NH, DQC = L::DQC, NKV = L::NKV;
  constexpr int kCB = D / 64;
  constexpr uint32_t kIdescS = idesc_f16(128, BK, false, false, kFp16);     // S, dP
  constexpr uint32_t kIdescKV = idesc_f16(128, NKV, true, true, kFp16);     // dV^T, dK^T
  constexpr uint32_t kIdescQ = idesc_f16(128, DQC, false, true, kFp16);     // dQ

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t qd_full[QS], qd_empty[QS], kv_full, kv_empty, sdp_full[NWG],
      sdp_free[NWG], pds_full[NWG], dq_full[NWG], dq_free, dkv_free;
  // K/V flags of the tile in each stage: bit 8 first tile of its run, bit 9 last
  __shared__ uint32_t qd_flags[QS];
  __shared__ uint32_t tmem_base;
  __shared__ int fail;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sQ0 = smem_u32(smem + L::kOffQ), sK = smem_u32(smem + L::kOffK),
                 sV = smem_u32(smem + L::kOffV), sP0 = smem_u32(smem + L::kOffP);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // zero the Q/dO stages once: with d = 64 their upper 64 columns stay zero
  if (D < 128) {
    for (int i = tid; i < static_cast<int>(QS * 2 * L::kQ / 16); i += blockDim.x)
      reinterpret_cast<uint4 *>(smem + L::kOffQ)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  if (warp == 5) tmem_alloc(&tmem_base, 512);
  if (tid == 0) {
    for (int i = 0; i < QS; ++i) {
      mbar_init(&qd_full[i], 32 * L::WPS);
      mbar_init(&qd_empty[i], 1);
    }
    mbar_init(&kv_full, 1);
    mbar_init(&kv_empty, 1);
    for (int w = 0; w < NWG; ++w) {
      mbar_init(&sdp_full[w], 1);
      mbar_init(&sdp_free[w], 128);
      mbar_init(&pds_full[w], 128);
      mbar_init(&dq_full[w], 1);
    }
    mbar_init(&dq_free, 128);
    mbar_init(&dkv_free, 128);
    fail = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tDQ = tmem_base + L::kTmDQ, tDV = tmem_base + L::kTmDV,
                 tDK = tmem_base + L::kTmDK;
  const int total = p.tile_off[p.h_k * (*p.nb)];
  const int C = p.bwd_chunk;
  auto same_run = [C](int ta, const TileDesc &a, int tb, const TileDesc &b) {
    return (a.hn & 0xffff) == (b.hn & 0xffff) && a.key0 == b.key0 && ta / C == tb / C;
  };

  if (warp < L::NPW) {
    // ------------------------------ producers ------------------------------
    constexpr int WPS = L::WPS, RW = L::RW, NJ = RW / 32;
    constexpr int kCPR = D / 8;           // 16-byte chunks per row
    constexpr int kRPI = 32 / kCPR;       // rows per warp instruction
    constexpr int kIJ = 32 / kRPI;        // warp instructions per 32 rows and tensor
    const int qs = warp / WPS, part = warp % WPS;   // stage, and rows [part RW, part RW + RW)
    TileSeq seq;
    seq.init(total, C);
    for (int k = 0; k < qs; ++k) seq.next();
    TileSeq prv;
    prv.init(total, C);
    for (int k = 0; k + 1 < qs; ++k) prv.next();
    const int oob_row = p.n * p.h_q;
    const uint16_t *gq = static_cast<const uint16_t *>(p.q);
    const uint16_t *gdo = static_cast<const uint16_t *>(p.dout);
    const uint64_t keep = l2_evict_last();
    const uint32_t stq = sQ0 + 2 * qs * L::kQ, stdo = stq + L::kQ;
    int li = qs;
    while (seq.valid()) {
      const TileDesc dc = load_desc(p, seq);
      TileSeq sn = seq;
      sn.next();
      const TileDesc dn = load_desc(p, sn);
      const TileDesc dp = li > 0 ? load_desc(p, prv) : TileDesc{0, 0, -1, -1};
      const int h = dc.hn & 0xffff, nrows = dc.hn >> 16;
      int rid[NJ];
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const int r = part * RW + j * 32 + lane;
        rid[j] = oob_row;
        if (r < nrows) {
          const int rr = dc.row0 + r;
          const int t = __ldg(p.q_list + dc.q_off + rr / p.g);
          rid[j] = t * p.h_q + h * p.g + rr % p.g;
        }
      }
      const bool first = li == 0 || !same_run(prv.tile(), dp, seq.tile(), dc);
      const bool last = !sn.valid() || !same_run(seq.tile(), dc, sn.tile(), dn);
      if (li >= QS) mbar_wait_sticky(&qd_empty[qs], ((li / QS) - 1) & 1, p.status, &fail);
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
#pragma unroll 4
        for (int k = 0; k < kIJ; ++k) {
          const int r32 = k * kRPI + lane / kCPR;          // row within this 32-row group
          const int id = __shfl_sync(0xffffffffu, rid[j], r32);
          const int r = part * RW + j * 32 + r32;          // tile row
          const int chunk = lane % kCPR;
          const bool in = id < oob_row;
          const int64_t off = in ? (int64_t)id * D + chunk * 8 : 0;
          const uint32_t so = sw128_offset(r, chunk, 128);
          cp_async16_hint(stq + so, gq + off, in ? 16u : 0u, keep);
          cp_async16_hint(stdo + so, gdo + off, in ? 16u : 0u, keep);
        }
      }
      cp_async_commit();
      if (lane == 0 && part == 0) qd_flags[qs] = (first ? 0x100u : 0u) | (last ? 0x200u : 0u);
      cp_async_wait_all();
      fence_proxy_async_smem();
      mbar_arrive(&qd_full[qs]);
      // this stage's next tile is li + QS; its predecessor is li + QS - 1
      prv = seq;
#pragma unroll
      for (int k = 0; k + 1 < QS; ++k) prv.next();
      seq = prv;
      seq.next();
      li += QS;
    }
  } else if (warp == 6) {
    // ------------------------------ K/V producer ------------------------------
    if (lane == 0) {
      const uint64_t keep = l2_evict_last();
      TileSeq seq;
      seq.init(total, C);
      int kv_n = 0, tprev = -1;
      TileDesc dprev{0, 0, -1, -1};
      while (seq.valid()) {
        const TileDesc dc = load_desc(p, seq);
        const int t = seq.tile(), h = dc.hn & 0xffff;
        if (tprev < 0 || !same_run(tprev, dprev, t, dc)) {
          if (kv_n >= 1) mbar_wait_sticky(&kv_empty, (kv_n - 1) & 1, p.status, &fail);
          mbar_arrive_expect_tx(&kv_full, 2u * L::kK);
#pragma unroll
          for (int cb = 0; cb < kCB; ++cb) {
            tma_load_3d_hint(sK + cb * BK * 128, &tm_k, cb * 64, h, dc.key0, &kv_full, keep);
            tma_load_3d_hint(sV + cb * BK * 128, &tm_v, cb * 64, h, dc.key0, &kv_full, keep);
          }
          ++kv_n;
        }
        tprev = t;
        dprev = dc;
        seq.next();
      }
    }
  } else if (warp == 4) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      TileSeq seq;
      seq.init(total, C);
      int n = 0;
      for (TileSeq c = seq; c.valid(); c.next()) ++n;
      // K/V flags of the tiles in flight (tiles i .. i + NWG), kept in registers by
      // tile index mod 4
      uint32_t fl0 = 0u, fl1 = 0u, fl2 = 0u, fl3 = 0u;
      auto fl_get = [&](int j) -> uint32_t {
        const int s = j & 3;
        return s == 0 ? fl0 : (s == 1 ? fl1 : (s == 2 ? fl2 : fl3));
      };
      auto fl_set = [&](int j, uint32_t f) {
        const int s = j & 3;
        if (s == 0) fl0 = f;
        else if (s == 1) fl1 = f;
        else if (s == 2) fl2 = f;
        else fl3 = f;
      };
      int s_kv = 0, runs = 0, dq_n = 0;
      int s_next = 0;    // next tile whose S/dP is to be issued
      int i_done = -1;   // last tile whose dV/dK/dQ MMAs (and K/V release) are issued
      // Issues S/dP of tiles s_next .. i_done + NWG.  Tile i_done + 1 is needed next,
      // so it is waited for; later tiles only if their Q/dO rows are in already.  A
      // tile that starts a new run waits until every earlier tile is issued, since
      // the K/V stage is released by the last tile of the previous run.
      auto try_issue = [&]() {
        while (s_next < n && s_next <= i_done + NWG) {
          const int j = s_next, qs = j % QS, w = j % NWG;
          const bool must = j == i_done + 1;
          if (must) mbar_wait_sticky(&qd_full[qs], (j / QS) & 1, p.status, &fail);
          else if (!mbar_test_wait(smem_u32(&qd_full[qs]), (j / QS) & 1)) break;
          const uint32_t f = qd_flags[qs];
          if ((f & 0x100u) && !must) break;
          fl_set(j, f);
          if (f & 0x100u) {
            mbar_wait_sticky(&kv_full, s_kv & 1, p.status, &fail);
            ++s_kv;
          }
          if (j >= NWG) mbar_wait_sticky(&sdp_free[w], ((j / NWG) - 1) & 1, p.status, &fail);
          // an aliased dQ occupies the S/dP columns until the epilogue has read it
          if (L::kDqAlias && dq_n > 0)
            mbar_wait_sticky(&dq_free, (dq_n - 1) & 1, p.status, &fail);
          tc_fence_after();
          const uint32_t stq = sQ0 + 2 * qs * L::kQ, stdo = stq + L::kQ;
          const uint32_t tSw = tmem_base + w * 2 * BK, tDPw = tSw + BK;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            mma_f16(tSw, desc_kmajor(stq, 128, kk), desc_kmajor(sK, BK, kk), kIdescS, kk > 0);
            mma_f16(tDPw, desc_kmajor(stdo, 128, kk), desc_kmajor(sV, BK, kk), kIdescS, kk > 0);
          }
          mma_commit(&sdp_full[w]);
          ++s_next;
        }
      };
      try_issue();
      for (int i = 0; i < n; ++i) {
        const int qs = i % QS, w = i % NWG;
        const uint32_t stq = sQ0 + 2 * qs * L::kQ, stdo = stq + L::kQ;
        const uint32_t sPw = sP0 + w * 2 * L::kP, sDSw = sPw + L::kP;
        // wait for P/dS(i), issuing S/dP of later tiles as their rows land
        {
          const uint32_t a = smem_u32(&pds_full[w]), par = (i / NWG) & 1;
          if (!mbar_test_wait(a, par)) {
            const uint64_t t0 = globaltimer_ns();
            while (!fail && !mbar_test_wait(a, par)) {
              try_issue();
              if (globaltimer_ns() - t0 > kWaitLimitNs) {
                fail = 1;
                set_status(p.status, NSA_DEVERR_TIMEOUT);
              }
            }
          }
        }
        const uint32_t f = fl_get(i);
        const bool first = (f & 0x100u) != 0;
        if (first) {
          if (runs > 0) mbar_wait_sticky(&dkv_free, (runs - 1) & 1, p.status, &fail);
          ++runs;
        }
        tc_fence_after();
        // dV^T += dO^T P and dK^T += Q^T dS (M = 128 rows of d per half, K = tile rows)
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t acc = (!first || ks > 0) ? 1u : 0u;
            mma_f16(tDV + hh * NKV, desc_mnmajor(stdo + hh * 2 * 128 * 128, 128, ks),
                    desc_mnmajor(sPw, 128, ks), kIdescKV, acc);
            mma_f16(tDK + hh * NKV, desc_mnmajor(stq + hh * 2 * 128 * 128, 128, ks),
                    desc_mnmajor(sDSw, 128, ks), kIdescKV, acc);
          }
        }
        mma_commit(&qd_empty[qs]);
        // dQ = dS K (M = tile rows, N = DQC columns of d per half, K = keys)
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          if (dq_n > 0) mbar_wait_sticky(&dq_free, (dq_n - 1) & 1, p.status, &fail);
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks)
            mma_f16(tDQ, desc_kmajor(sDSw, 128, ks),
                    desc_mnmajor(sK + hh * 2 * BK * 128, BK, ks), kIdescQ, ks > 0);
          mma_commit(&dq_full[w]);
          ++dq_n;
        }
        if (f & 0x200u) mma_commit(&kv_empty);
        i_done = i;
        try_issue();
      }
    }
  } else if (warp >= 8 && ((warp - 8) >> 2) < NWG) {
    // ----------------------------- compute warpgroups -----------------------------
    const int wg = (warp - 8) >> 2;
    const int row = (tid - 256) & 127;                      // tile row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem_base + wg * 2 * BK, tDP = tS + BK;
    const uint32_t sP = sP0 + wg * 2 * L::kP, sDS = sP + L::kP;
    const uint64_t stream = l2_evict_first();
    const float kLog2e = 1.4426950408889634f;
    TileSeq seq;
    seq.init(total, C);
    if (wg == 1) seq.next();
    // keys [lo, lim] of the block are visible to the row (lim < 0: no row): the causal
    // limit and the start of a sliding window (0 without one)
    auto row_meta = [&](const TileDesc &d, int &lim, int &lo, float &lse2, float &dval) {
      const int nrows = d.hn >> 16, h = d.hn & 0xffff;
      lim = -1;
      lo = 0;
      lse2 = 0.f;
      dval = 0.f;
      if (row < nrows) {
        const int rr = d.row0 + row;
        const int t = __ldg(p.q_list + d.q_off + rr / p.g);
        const int hq = h * p.g + rr % p.g;
        lim = min(BK - 1, t - d.key0);
        if (kWin) lo = max(0, t - p.window + 1 - d.key0);
        lse2 = __ldg(p.lse_in + (int64_t)hq * p.n + t) * kLog2e;
        dval = __ldg(p.dstat + (int64_t)hq * p.n + t);
      }
    };
    TileDesc dsc = load_desc(p, seq);
    int lim = -1, lo = 0;
    float lse2 = 0.f, dval = 0.f;
    if (seq.valid()) row_meta(dsc, lim, lo, lse2, dval);
    int dqw = 0;                                 // dQ halves this warpgroup has consumed
    for (int i = wg; seq.valid(); i += NWG) {
      const int tile = seq.tile();
      TileSeq nseq = seq;                        // the CTA's next tile (ends a run?)
      nseq.next();
      TileSeq mseq = nseq;                       // this warpgroup's next tile
#pragma unroll
      for (int k = 1; k < NWG; ++k) mseq.next();
      const TileDesc ndsc = load_desc(p, nseq);
      const TileDesc mdsc = NWG == 1 ? ndsc : load_desc(p, mseq);
      mbar_wait_sticky(&sdp_full[wg], (i / NWG) & 1, p.status, &fail);
      tc_fence_after();
      // ---- P and dS of this row, written in 16 bits as MMA operands ----
      // A warp whose rows all see the whole block skips the mask.  Rows past the
      // tile's end take that path too: their Q and dO rows are zero, so they add
      // nothing to dV, dK or a dQ row anyone reads.  dS uses the 16-bit P the MMAs see.
      const bool full = __all_sync(0xffffffffu, lim < 0 || (lim >= BK - 1 && lo <= 0));
#pragma unroll
      for (int c = 0; c < BK / 32; ++c) {
        float sv[32], dp[32];
        tmem_ld32(tS + lane_off + c * 32, sv);
        tmem_ld32(tDP + lane_off + c * 32, dp);
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int ii = c * 32 + j;
          float p0 = ex2_approx(fmaf(sv[j], p.scale_log2, -lse2));
          float p1 = ex2_approx(fmaf(sv[j + 1], p.scale_log2, -lse2));
          if (!full) {
            p0 = (ii <= lim && ii >= lo) ? p0 : 0.f;
            p1 = (ii + 1 <= lim && ii + 1 >= lo) ? p1 : 0.f;
          }
          pp[j / 2] = pack2<kFp16>(p0, p1);
          const float2 pr = unpack2<kFp16>(pp[j / 2]);
          dd[j / 2] = pack2<kFp16>(pr.x * (dp[j] - dval), pr.y * (dp[j + 1] - dval));
        }
        st_row_packed(sP, row, c * 4, pp);
        st_row_packed(sDS, row, c * 4, dd);
      }
      if constexpr (BK < 64) {   // zero the unused half of the swizzle atom read by N = 64
        float z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = 0.f;
        st_row_chunks<kFp16>(sP, row, 4, z);
        st_row_chunks<kFp16>(sDS, row, 4, z);
      }
      tc_fence_before();
      if (!L::kDqAlias) mbar_arrive(&sdp_free[wg]);
      fence_proxy_async_smem();
      mbar_arrive(&pds_full[wg]);
      // this warpgroup's next tile's row metadata: its loads overlap the MMAs and the epilogue
      int nlim = -1, nlo = 0;
      float nlse2 = 0.f, ndval = 0.f;
      if (mseq.valid()) row_meta(mdsc, nlim, nlo, nlse2, ndval);

      // ---- dQ epilogue: TMEM -> 16 bits -> this warp's staging slots -> TMA
      //      stores.  The slots lie in this warpgroup's P buffer (and, with a single
      //      dQ pass, its dS buffer too): free once the dQ MMA of this tile completed ----
      constexpr int kSlots = (NH == 1 ? 2 : 1) * static_cast<int>(L::kP / (4 * 4096));
      const uint32_t stg = sP + (warp & 3) * kSlots * 4096u;
      int used = 0;                              // stores issued from this warp's slots
#pragma unroll
      for (int hh = 0; hh < NH; ++hh) {
        mbar_wait_sticky(&dq_full[wg], dqw & 1, p.status, &fail);
        ++dqw;
        tc_fence_after();
#pragma unroll
        for (int cb = 0; cb < DQC / 64; ++cb) {
          float v[64];
          tmem_ld64(tDQ + lane_off + cb * 64, v);
          if (cb == DQC / 64 - 1) {
            tc_fence_before();
            mbar_arrive(&dq_free);
            if (L::kDqAlias && hh == NH - 1) mbar_arrive(&sdp_free[wg]);
          }
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 64; j += 2) pk[j / 2] = pack2<kFp16>(v[j], v[j + 1]);
          const uint32_t slot = stg + (used % kSlots) * 4096u;
          if (lane == 0 && used >= kSlots) bulk_wait_read_all();   // the slot's last store
          __syncwarp();
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            const uint32_t so = sw128_offset(lane, q4, 32);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(slot + so),
                         "r"(pk[q4 * 4]), "r"(pk[q4 * 4 + 1]), "r"(pk[q4 * 4 + 2]),
                         "r"(pk[q4 * 4 + 3])
                         : "memory");
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d_hint(&tm_dq, slot, hh * 128 + cb * 64,
                              tile * kTileRows + (warp & 3) * 32, stream);
            bulk_commit();
          }
          ++used;
        }
      }
      // the staging slots are this warpgroup's next P/dS rows, written by all four of
      // its warps: every warp's stores must have been read first
      if (lane == 0) bulk_wait_read_all();
      named_bar_sync(1 + wg, 128);

      // ---- end of a run: dK, dV partials out (fp32), one slot per (segment, chunk) ----
      const bool last = !nseq.valid() || !same_run(tile, dsc, nseq.tile(), ndsc);
      if (last) {
        const int seg = p.tseg[tile];
        const int slot = p.part_off[seg] + tile / C - p.tile_off[seg] / C;
        float *dst = p.dkvbuf + (int64_t)slot * 2 * BK * D;
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          const int dd = hh * 128 + row;        // d index of this TMEM lane
#pragma unroll
          for (int c = 0; c < BK / 32; ++c) {
            float v[32], w[32];
            tmem_ld32(tDV + hh * NKV + lane_off + c * 32, v);
            tmem_ld32(tDK + hh * NKV + lane_off + c * 32, w);
            if (dd < D) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                dst[(int64_t)(c * 32 + j) * D + dd] = v[j];
                dst[(int64_t)BK * D + (c * 32 + j) * D + dd] = w[j];
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&dkv_free);
      }
      seq = mseq;
      dsc = mdsc;
      lim = nlim;
      lo = nlo;
      lse2 = nlse2;
      dval = ndval;
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem_base, 512);
}

// dq[t, hq] = scale * sum_k dQ_part[prow[h, t, k] + j]; one warp per row.
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
    const int32_t pr = p.prow[((int64_t)h * p.n + t) * p.topk + lane];
    if (pr >= 0) row = (int64_t)pr + j;
  }
  const uint16_t *buf = reinterpret_cast<const uint16_t *>(p.dqbuf);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  constexpr int kBatch = 16;   // partial rows in flight per lane
  for (int k0 = 0; k0 < p.topk; k0 += kBatch) {
    uint32_t u[kBatch][E / 2];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t r = __shfl_sync(0xffffffffu, row, (k0 + b) & 31);
      const bool ok = k0 + b < p.topk && r >= 0;
      const uint16_t *src = buf + (ok ? r : 0) * D + lane * E;
      if constexpr (E == 2) {
        u[b][0] = ok ? __ldcs(reinterpret_cast<const unsigned int *>(src)) : 0u;
      } else if constexpr (E == 4) {
        const uint2 x = ok ? __ldcs(reinterpret_cast<const uint2 *>(src)) : make_uint2(0u, 0u);
        u[b][0] = x.x; u[b][1] = x.y;
      } else {
        const uint4 x = ok ? __ldcs(reinterpret_cast<const uint4 *>(src))
                           : make_uint4(0u, 0u, 0u, 0u);
        u[b][0] = x.x; u[b][1] = x.y; u[b][2] = x.z; u[b][3] = x.w;
      }
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
#pragma unroll
      for (int e = 0; e < E / 2; ++e) {
        const float2 f = unpack2<kFp16>(u[b][e]);
        acc[2 * e] += f.x;
        acc[2 * e + 1] += f.y;
      }
  }
  uint16_t *dst = static_cast<uint16_t *>(p.dq) + wid * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    *reinterpret_cast<uint32_t *>(dst + e) = pack2<kFp16>(acc[e] * p.scale, acc[e + 1] * p.scale);
}

// dk, dv of eight keys of one (KV head, block): sums of the segment's partials
// (zeros if none).  Block (seg, y) takes keys [8 y, 8 y + 8); each thread four
// consecutive d elements of one key, reading eight partials at a time.
constexpr int kDkvKeys = 8;
template <int D, int BK, bool kFp16>
__global__ void __launch_bounds__(kDkvKeys * D / 4) bwd_dkv_kernel(Params p) {
  const int nb = *p.nb;
  const int seg = blockIdx.x;
  if (seg >= p.h_k * nb) return;
  const int h = seg / nb, gb = seg - h * nb;
  const int s = upper_index(p.blk_start, p.num_seqs + 1, gb);
  const int b = gb - p.blk_start[s];
  const int key0 = p.cu[s] + b * BK;
  const int nkeys = min(BK, p.cu[s + 1] - key0);
  const int key = blockIdx.y * kDkvKeys + static_cast<int>(threadIdx.x) / (D / 4);
  const int x = (static_cast<int>(threadIdx.x) % (D / 4)) * 4;
  if (key >= nkeys) return;
  const int c0 = p.part_off[seg], c1 = p.part_off[seg + 1];
  const float *base = p.dkvbuf + (int64_t)key * D + x;
  float4 av = make_float4(0.f, 0.f, 0.f, 0.f), ak = av;
  for (int c = c0; c < c1; c += 8) {
    float4 v[8], k[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const bool ok = c + u < c1;
      const float *src = base + (int64_t)(ok ? c + u : c0) * 2 * BK * D;
      v[u] = ok ? __ldg(reinterpret_cast<const float4 *>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
      k[u] = ok ? __ldg(reinterpret_cast<const float4 *>(src + BK * D))
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      av.x += v[u].x; av.y += v[u].y; av.z += v[u].z; av.w += v[u].w;
      ak.x += k[u].x; ak.y += k[u].y; ak.z += k[u].z; ak.w += k[u].w;
    }
  }
  uint16_t *dk = static_cast<uint16_t *>(p.dk), *dv = static_cast<uint16_t *>(p.dv);
  const int64_t o = ((int64_t)(key0 + key) * p.h_k + h) * D + x;
  *reinterpret_cast<uint2 *>(dk + o) =
      make_uint2(pack2<kFp16>(ak.x * p.scale, ak.y * p.scale),
                 pack2<kFp16>(ak.z * p.scale, ak.w * p.scale));
  *reinterpret_cast<uint2 *>(dv + o) = make_uint2(pack2<kFp16>(av.x, av.y), pack2<kFp16>(av.z, av.w));
}

// ---------------------------------------------------------------------------
// Host-side dispatch
// ---------------------------------------------------------------------------
bool make_kv_maps(const Params &p, CUtensorMap *mk, CUtensorMap *mv);
bool make_rows_map(const Params &p, void *base, int64_t max_tiles, CUtensorMap *m);

template <int D, int BK, bool kFp16>
static cudaError_t run_bwd(const Params &p, int num_sms, int64_t max_tiles, cudaStream_t stream,
                           void (*mark)(int, cudaStream_t, bool)) {
  using L = BwdCfg<D, BK>;
  CUtensorMap mk, mv, mdq;
  if (!make_kv_maps(p, &mk, &mv) || !make_rows_map(p, p.dqbuf, max_tiles, &mdq))
    return cudaErrorInvalidValue;
  const int64_t rows = static_cast<int64_t>(p.n) * p.h_q;
  int grid = num_sms < kMaxBwdCtas ? num_sms : kMaxBwdCtas;
  mark(7, stream, true);
  bwd_pre_kernel<D, kFp16><<<static_cast<unsigned>((rows + 31) / 32), 256, 0, stream>>>(p);
  bwd_parts_kernel<<<1, 1024, 0, stream>>>(p);
  mark(7, stream, false);
  const uint32_t smem = L::kBytes;
  auto kern = p.window > 0 ? bwd_main_kernel<D, BK, kFp16, true>
                            : bwd_main_kernel<D, BK, kFp16, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  mark(8, stream, true);
  kern<<<static_cast<unsigned>(grid), L::kThreads, smem, stream>>>(mk, mv, mdq, p);
  mark(8, stream, false);
  // dK/dV first: the two reductions are independent, and dk/dv are then final while
  // the larger dQ reduction runs (the end of mark 10 is where a caller may start
  // copying them)
  mark(10, stream, true);
  bwd_dkv_kernel<D, BK, kFp16>
      <<<dim3(static_cast<unsigned>(p.h_k * p.nb_max), BK / kDkvKeys), kDkvKeys * D / 4, 0,
         stream>>>(p);
  mark(10, stream, false);
  mark(9, stream, true);
  bwd_dq_kernel<D, kFp16><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(p);
  mark(9, stream, false);
  return cudaGetLastError();
}

template <int D, bool kFp16>
static cudaError_t run_bwd_bk(const Params &p, int num_sms, int64_t max_tiles, cudaStream_t s,
                              void (*mark)(int, cudaStream_t, bool)) {
  switch (p.block) {
    case 32: return run_bwd<D, 32, kFp16>(p, num_sms, max_tiles, s, mark);
    case 64: return run_bwd<D, 64, kFp16>(p, num_sms, max_tiles, s, mark);
    case 128:
      if constexpr (D == 256) return cudaErrorInvalidValue;
      else return run_bwd<D, 128, kFp16>(p, num_sms, max_tiles, s, mark);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd(const Params &p, int num_sms, int64_t max_tiles, cudaStream_t s,
                       void (*mark)(int, cudaStream_t, bool)) {
  const bool f16 = p.dtype == NSA_FP16;
  switch (p.d) {
    case 64: return f16 ? run_bwd_bk<64, true>(p, num_sms, max_tiles, s, mark)
                        : run_bwd_bk<64, false>(p, num_sms, max_tiles, s, mark);
    case 128: return f16 ? run_bwd_bk<128, true>(p, num_sms, max_tiles, s, mark)
                         : run_bwd_bk<128, false>(p, num_sms, max_tiles, s, mark);
    case 256: return f16 ? run_bwd_bk<256, true>(p, num_sms, max_tiles, s, mark)
                         : run_bwd_bk<256, false>(p, num_sms, max_tiles, s, mark);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nsa
