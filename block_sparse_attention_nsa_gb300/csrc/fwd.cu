// fwd.cu -- forward of NSA selected attention on sm_103a.
//
// Loop order follows "FSA: An Alternative Efficient Implementation of Native
// Sparse Attention Kernel" (key design 1): the outer loop is over KV blocks, the
// inner one over 128-row tiles of the query rows (token, query head) that selected
// the block, so the MMA's M dimension is filled by gathered queries and no
// GQA-group padding is needed.  Tiles come from (KV head, wave, block)
// sub-segments of the index: a wave is a window of consecutive tokens, so the
// rows of one wave are finished before the next wave starts.
//
//   fwd_main  : per tile, S = Q K_b^T (tcgen05, TMEM accumulator, M = 128,
//               N = B_K); masked row max m and P = exp2(S*scale*log2e - m) in
//               registers, P written back to TMEM in 16 bits; O = P V_b (tcgen05
//               with A = P read from TMEM, N = d).  The unnormalised partial O of
//               every row and its (m, l = fp32 sum of P) go to the compact buffer
//               (key design 2), one 128-row block per tile, by TMA tensor stores.
//   fwd_merge : per (token, query head), the <= T partials are combined with
//               log-sum-exp weights into out and lse.  Carrying (m, l) with each
//               partial replaces the separate statistics kernel of key design 4:
//               every partial is rescaled once, at merge time, by exp2(m - M).
#include "common.cuh"

namespace nsa {

// Pipeline depths per (d, B_K), bounded by 227 KB of shared memory: Q stages,
// K/V stages and output staging slots per softmax warpgroup (one 64-column block
// of 128 rows each; two let a warpgroup fill one while the TMA store of the other
// drains).  TMEM (512 columns): two S slots of B_K columns (P, in 16 bits,
// overwrites the first B_K / 2 columns of its S slot) and OS fp32 O accumulators
// of d columns.
__host__ __device__ constexpr int fwd_qs(int d, int bk) {
  return d == 64 ? 4 : (d == 128 ? 4 : (bk == 128 ? 1 : 2));
}
__host__ __device__ constexpr int fwd_kvs(int d, int bk) {
  return d == 64 ? 2 : (d == 128 ? (bk == 128 ? 1 : 2) : (bk <= 32 ? 2 : 1));
}
__host__ __device__ constexpr int fwd_ss(int d) { return d == 64 ? 2 : 1; }
__host__ __device__ constexpr int fwd_os(int d, int bk) { return 2 * bk + 2 * d <= 512 ? 2 : 1; }

template <int D, int BK>
struct FwdSmem {
  static constexpr int QS = fwd_qs(D, BK), KVS = fwd_kvs(D, BK), SS = fwd_ss(D),
                       OS = fwd_os(D, BK);
  static constexpr int NPW = QS < 4 ? QS : 4;   // Q producer warps (one per stage or more)
  static_assert(QS % NPW == 0, "each Q stage needs a single producer warp");
  // each of the two MMA threads consumes every other tile: with an even number of Q
  // stages each stage belongs to one thread; a single stage is handled explicitly
  static_assert(QS % 2 == 0 || QS == 1, "Q stages: even, or one");
  static constexpr uint32_t kQ = 128u * D * 2u;            // one Q stage
  static constexpr uint32_t kK = uint32_t(BK) * D * 2u;     // one K (or V) stage
  static constexpr uint32_t kStg = 128u * 64u * 2u;         // staging of one warpgroup
  static constexpr uint32_t kStgW = 32u * 64u * 2u;         // one warp's staging slot
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + QS * kQ;
  static constexpr uint32_t kOffV = kOffK + KVS * kK;
  static constexpr uint32_t kOffStg = kOffV + KVS * kK;
  static constexpr uint32_t kBytes = kOffStg + 2 * SS * kStg + 1024;   // + alignment slack
  static_assert(kBytes <= 227u * 1024u, "shared memory budget");
  static_assert(2 * BK + OS * D <= 512, "TMEM budget");
  static constexpr uint32_t kTmemCols = 512;
};

// warps 0-3 Q producers, warps 4 and 7 MMA issuers, warp 5 TMEM owner, warp 6 K/V
// producer, warps 8-11 / 12-15 two softmax WGs
constexpr int kFwdThreads = 512;

// Persistent, warp-specialised forward main kernel (one CTA per SM).
//   warps 0-3: producers (as many as Q stages, at most 4) -- warp w gathers the
//     Q rows of tiles w, w + NPW, ... by
//     cp.async (16-byte chunks, a warp instruction covering 256 / d whole rows,
//     so reads are fully coalesced) into the 128-byte-swizzled operand layout,
//     waits for its own copies and arrives; a Q stage is released (by the softmax
//     warpgroup of its tile) as soon as the S MMA that reads it has completed;
//   warp 6 (one thread): K_b and V_b by TMA (3-D tensor maps, once per change of
//     (KV head, block));
//   warps 4 and 7 (one thread each): tcgen05 MMAs of the even and of the odd
//     tiles, S(i) = Q K^T into TMEM slot i % 2 and O(i) = P V into an O
//     accumulator, issued as S(i), O(i), S(i + 2), ... by each;
//   warps 8-11 / 12-15: softmax of even / odd tiles (row max, exp2, P in 16 bits
//     back to TMEM, fp32 row sum) and their epilogue (O from TMEM to 16 bits,
//     staged one 64-column block at a time and written by TMA tensor stores to
//     the tile's 128 rows of the compact buffer; (m, l) per row).
// mbarriers hand each buffer between roles; every wait is bounded.
// kWin: the sliding window's lower key bound is applied (p.window > 0); without it
// the bound is compiled out.
template <int D, int BK, bool kFp16, bool kWin>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_main_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, Params p) {
  using L = FwdSmem<D, BK>;
  constexpr int QS = L::QS, KVS = L::KVS, OS = L::OS;
  constexpr int kCB = D / 64;                      // 64-column blocks per row
  constexpr uint32_t kIdescS = idesc_f16(128, BK, false, false, kFp16);
  constexpr uint32_t kIdescO = idesc_f16(128, D, false, true, kFp16);

  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t q_full[QS], q_empty[QS], kv_full[KVS], kv_empty[KVS], s_full[2],
      p_full[2], o_full[2], o_free[OS];
  __shared__ uint32_t tmem_base;
  __shared__ int fail;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t sQ0 = smem_u32(smem + L::kOffQ), sK0 = smem_u32(smem + L::kOffK),
                 sV0 = smem_u32(smem + L::kOffV), sStg0 = smem_u32(smem + L::kOffStg);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 5) tmem_alloc(&tmem_base, L::kTmemCols);
  if (tid == 0) {
    for (int i = 0; i < QS; ++i) { mbar_init(&q_full[i], 32); mbar_init(&q_empty[i], 1); }
    // kv_empty: one arrival from each MMA thread
    for (int i = 0; i < KVS; ++i) { mbar_init(&kv_full[i], 1); mbar_init(&kv_empty[i], 2); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 128);
      mbar_init(&o_full[i], 1);
    }
    for (int i = 0; i < OS; ++i) mbar_init(&o_free[i], 128);
    fail = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS0 = tmem_base, tO0 = tmem_base + 2 * BK;
  const int total = p.wtile_off[p.nsub];

  if (warp < L::NPW) {
    // ------------------------------ producer ------------------------------
    // Warp w gathers whole tiles w, w + NPW, w + 2 NPW, ... of this CTA: it waits
    // for its own copies of a tile, fences them for the tensor core and arrives,
    // so a tile's readiness never depends on the issue of later tiles.  NPW
    // divides QS, so every Q stage has exactly one producer warp and no waiter on
    // a stage's barriers can run two phases ahead.
    constexpr int NPW = L::NPW;
    constexpr int kCPR = D / 8;           // 16-byte chunks per row
    constexpr int kRPI = 32 / kCPR;       // rows per warp instruction
    constexpr int kIns = 128 / kRPI;      // warp instructions per tile
    TileSeq seq;
    seq.init(total, p.fwd_chunk);
    for (int k = 0; k < warp; ++k) seq.next();
    const int oob_row = p.n * p.h_q;
    // rid[j] = global Q row of tile row 32 j + lane (oob_row for padding rows)
    auto tile_rids = [&](const TileDesc &d, int (&rid)[4]) {
      const int h = d.hn & 0xffff, nrows = d.hn >> 16;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = j * 32 + lane;
        rid[j] = oob_row;
        if (r < nrows) {
          const int rr = d.row0 + r;
          const int t = __ldg(p.q_list + d.q_off + rr / p.g);
          rid[j] = t * p.h_q + h * p.g + rr % p.g;
        }
      }
    };
    const uint16_t *gq = static_cast<const uint16_t *>(p.q);
    const uint64_t keep = l2_evict_last();    // Q rows are gathered ~T times each
    int li = warp;
    while (seq.valid()) {
      const TileDesc dc = load_desc(p, seq);
      int rid[4];
      tile_rids(dc, rid);
      const int qs = li % QS;
      if (li >= QS) mbar_wait_sticky(&q_empty[qs], ((li / QS) - 1) & 1, p.status, &fail);
      const uint32_t stage = sQ0 + qs * L::kQ;
#pragma unroll
      for (int j = 0; j < 4; ++j) {              // tile rows 32 j .. 32 j + 31
#pragma unroll 4
        for (int k = 0; k < kIns / 4; ++k) {
          const int r = (j * (kIns / 4) + k) * kRPI + lane / kCPR;   // this lane's row
          const int id = __shfl_sync(0xffffffffu, rid[j], r & 31);
          const int chunk = lane % kCPR;
          const bool in = id < oob_row;
          cp_async16_hint(stage + sw128_offset(r, chunk, 128),
                          gq + (in ? (int64_t)id * D + chunk * 8 : 0), in ? 16u : 0u, keep);
        }
      }
      cp_async_commit();
      cp_async_wait_all();
      fence_proxy_async_smem();
      mbar_arrive(&q_full[qs]);
#pragma unroll
      for (int k = 0; k < NPW; ++k) seq.next();   // this warp's next tile: li + NPW
      li += NPW;
    }
  } else if (warp == 6) {
    // --------------------------- K/V producer -----------------------------
    // A warp of its own: its waits on kv_empty must not hold back the Q
    // producers, whose q_full arrivals lag their copies by QS - 1 tiles.
    if (lane == 0) {
      const uint64_t keep = l2_evict_last();    // a block's K/V serve all its tiles
      TileSeq seq;
      seq.init(total, p.fwd_chunk);
      int kv_n = 0, prev_h = -1, prev_key0 = -1;
      TileDesc dc = load_desc(p, seq);
      TileSeq seq1 = seq;
      seq1.next();
      TileDesc dn = load_desc(p, seq1);
      while (seq.valid()) {
        TileSeq seq2 = seq1;
        seq2.next();
        const TileDesc dnn = load_desc(p, seq2);
        const int h = dc.hn & 0xffff;
        if (h != prev_h || dc.key0 != prev_key0) {
          const int ks = kv_n % KVS;
          if (kv_n >= KVS)
            mbar_wait_sticky(&kv_empty[ks], ((kv_n / KVS) - 1) & 1, p.status, &fail);
          mbar_arrive_expect_tx(&kv_full[ks], 2u * L::kK);
#pragma unroll
          for (int cb = 0; cb < kCB; ++cb) {
            tma_load_3d_hint(sK0 + ks * L::kK + cb * BK * 128, &tm_k, cb * 64, h, dc.key0,
                             &kv_full[ks], keep);
            tma_load_3d_hint(sV0 + ks * L::kK + cb * BK * 128, &tm_v, cb * 64, h, dc.key0,
                             &kv_full[ks], keep);
          }
          ++kv_n;
          prev_h = h;
          prev_key0 = dc.key0;
        }
        seq = seq1;
        seq1 = seq2;
        dc = dn;
        dn = dnn;
      }
    }
  } else if ((warp == 4 || warp == 7) && lane == 0) {
    // ------------------------------ MMA issuers ------------------------------
    // Thread w (warp 4 for w = 0, warp 7 for w = 1) issues the MMAs of the tiles of
    // softmax warpgroup w, i = w, w + 2, ...: S(i) into S slot w, then, once P(i) is
    // in, O(i); S(i + 2) follows O(i) in the same thread, so the tensor pipe
    // executes them in order (S(i + 2) overwrites the columns P(i) was read from).
    // The two threads' MMAs interleave on the tensor pipe, and one thread's waits
    // for its warpgroup are covered by the other's issue.  Both walk every tile of
    // the CTA to follow the K/V loads; a load is released (kv_empty, count 2) by
    // each thread after its last MMA that reads it, or at once if it has none.
    const int w = warp == 4 ? 0 : 1;
    constexpr uint32_t kHiK = sdesc_hi_sw128(1024);   // K-major Q, K and MN-major V
    uint32_t lo_q[QS], lo_k[KVS], lo_v[KVS];
#pragma unroll
    for (int j = 0; j < QS; ++j) lo_q[j] = sdesc_lo_sw128(sQ0 + j * L::kQ, 16);
#pragma unroll
    for (int j = 0; j < KVS; ++j) {
      lo_k[j] = sdesc_lo_sw128(sK0 + j * L::kK, 16);
      lo_v[j] = sdesc_lo_sw128(sV0 + j * L::kK, BK * 128);
    }
    const uint32_t tSw = tS0 + w * BK;
    // descriptors of tiles i, i + 1 and i + 2 (loaded two tiles ahead)
    TileSeq seq;
    seq.init(total, p.fwd_chunk);
    TileSeq s2 = seq;
    s2.next();
    TileDesc dc = load_desc(p, seq);
    TileDesc dn = load_desc(p, s2);
    s2.next();
    TileDesc dnn = load_desc(p, s2);
    int m = -1;              // K/V load of the current run (load m fills stage m % KVS)
    bool own = false;        // this thread has issued an MMA that reads load m
    int prev_h = -1, prev_key0 = -1;
    for (int i = 0; seq.valid(); ++i) {
      const int h = dc.hn & 0xffff;
      if (h != prev_h || dc.key0 != prev_key0) {   // a new K/V load
        ++m;
        own = false;
        prev_h = h;
        prev_key0 = dc.key0;
      }
      TileSeq s1 = seq;
      s1.next();
      const bool last = !s1.valid() || (dn.hn & 0xffff) != h || dn.key0 != dc.key0;
      const int ks = m % KVS;
      const uint32_t kv_par = (m / KVS) & 1;
      if ((i & 1) == w) {
        if (!own) {
          mbar_wait_sticky(&kv_full[ks], kv_par, p.status, &fail);
          own = true;
        }
        const int qs = i % QS, os = i % OS;
        if constexpr (QS == 1) {
          // A single Q stage alternates between the two threads: wait until the other
          // thread's tile i - 1 has consumed its fill, so that the wait below cannot
          // be met by the phase of tile i - 2
          if (i >= 1) mbar_wait_sticky(&s_full[1 - w], ((i - 1) >> 1) & 1, p.status, &fail);
        }
        mbar_wait_sticky(&q_full[qs], (i / QS) & 1, p.status, &fail);
        tc_fence_after();
        uint32_t aq = lo_q[0], bk = lo_k[0], bv = lo_v[0];
#pragma unroll
        for (int j = 1; j < QS; ++j) aq = qs == j ? lo_q[j] : aq;
#pragma unroll
        for (int j = 1; j < KVS; ++j) {
          bk = ks == j ? lo_k[j] : bk;
          bv = ks == j ? lo_v[j] : bv;
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_f16(tSw, sdesc_join(aq + (kmajor_step(128, kk) >> 4), kHiK),
                  sdesc_join(bk + (kmajor_step(BK, kk) >> 4), kHiK), kIdescS, kk > 0);
        mma_commit(&s_full[w]);   // the softmax warpgroup then releases Q stage qs
        mbar_wait_sticky(&p_full[w], (i >> 1) & 1, p.status, &fail);
        if (i >= OS) mbar_wait_sticky(&o_free[os], ((i / OS) - 1) & 1, p.status, &fail);
        tc_fence_after();
        const uint32_t tOd = tO0 + os * D;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          mma_f16_ts(tOd, tSw + kk * 8, sdesc_join(bv + (mnmajor_step(kk) >> 4), kHiK),
                     kIdescO, kk > 0);
        mma_commit(&o_full[w]);
      }
      if (last) {
        if (own) {
          mma_commit(&kv_empty[ks]);
        } else {
          mbar_wait_sticky(&kv_full[ks], kv_par, p.status, &fail);
          mbar_arrive(&kv_empty[ks]);
        }
      }
      seq = s1;
      dc = dn;
      dn = dnn;
      s2.next();
      dnn = load_desc(p, s2);
    }
  } else if (warp >= 8) {
    // ------------------------- softmax + epilogue -------------------------
    const int wg = (warp - 8) >> 2;
    const int row = tid - 256 - wg * 128;                  // tile row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    constexpr int SS = L::SS;
    const uint32_t stg = sStg0 + (warp - 8) * SS * L::kStgW;
    const uint64_t stream = l2_evict_first();   // partials are read once, by the merge
    TileSeq seq;
    seq.init(total, p.fwd_chunk);
    if (wg == 1) seq.next();
    // descriptor and key range of this warpgroup's next tile, loaded one tile early:
    // keys [lo, lim] of the block are visible to the row (lim < 0: no row); lim is the
    // causal limit, lo the start of a sliding window (0 without one)
    auto tile_lim = [&](const TileDesc &d) {
      const int nrows = d.hn >> 16;
      if (row >= nrows) return make_int2(-1, 0);
      const int t = __ldg(p.q_list + d.q_off + (d.row0 + row) / p.g);
      const int lo = kWin ? max(0, t - p.window + 1 - d.key0) : 0;
      return make_int2(min(BK - 1, t - d.key0), lo);
    };
    TileDesc dsc = load_desc(p, seq);
    int2 lr = seq.valid() ? tile_lim(dsc) : make_int2(-1, 0);
    int lim = lr.x, lo = lr.y;
    TileSeq nseq = seq;
    nseq.next();
    nseq.next();
    TileDesc ndsc = load_desc(p, nseq);
    int n_cb = 0;                                 // column blocks stored so far
    for (int i = wg; seq.valid(); i += 2) {
      const int tile = seq.tile();
      const int nrows = dsc.hn >> 16;
      const bool row_in = row < nrows;
      const int os = i % OS;
      mbar_wait_sticky(&s_full[i & 1], (i >> 1) & 1, p.status, &fail);
      // S(i) is complete, so its MMAs have read Q stage i % QS: release it
      if (row == 0) mbar_arrive(&q_empty[i % QS]);
      tc_fence_after();
      const uint32_t tS = tS0 + (i & 1) * BK + lane_off;
      float lsum = 0.f, m2 = 0.f;
      if constexpr (BK == 128) {
        // two passes over 32-column chunks (128 scores do not stay in registers)
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < BK / 32; ++c) {
          float sv[32];
          tmem_ld32(tS + c * 32, sv);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j <= lim && c * 32 + j >= lo) mx = fmaxf(mx, sv[j]);
        }
        m2 = row_in ? mx * p.scale_log2 : 0.f;
#pragma unroll
        for (int c = 0; c < BK / 32; ++c) {
          float sv[32];
          tmem_ld32(tS + c * 32, sv);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int ii = c * 32 + j;
            const float p0 =
                (ii <= lim && ii >= lo) ? ex2_approx(fmaf(sv[j], p.scale_log2, -m2)) : 0.f;
            const float p1 = (ii + 1 <= lim && ii + 1 >= lo)
                                 ? ex2_approx(fmaf(sv[j + 1], p.scale_log2, -m2))
                                 : 0.f;
            lsum += p0 + p1;                    // fp32 row sum (exact lse)
            pk[j / 2] = pack2<kFp16>(p0, p1);   // P rounded to 16 bits for the PV MMA
          }
          // 32 P values of this chunk -> 16 TMEM columns; they overwrite S columns
          // [16 c, 16 c + 16), which this thread has already read.
          tmem_st16(tS + c * 16, pk);
        }
      } else {
        // all B_K scores of the row in registers: one TMEM load, one wait
        float sv[BK];
        if constexpr (BK == 64) {
          tmem_ld64(tS, sv);
        } else {
          tmem_ld32(tS, sv);
        }
        // Only rows of a tile of the token's own block (or of a window's first block)
        // need a mask; a warp whose rows all see the whole block takes the unmasked
        // path.  Eight independent max / sum chains keep the dependent latency short.
        const bool full = __all_sync(0xffffffffu, !row_in || (lim >= BK - 1 && lo <= 0));
        float mxs[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) mxs[j] = -INFINITY;
        if (full) {
#pragma unroll
          for (int j = 0; j < BK; ++j) mxs[j & 7] = fmaxf(mxs[j & 7], sv[j]);
        } else {
#pragma unroll
          for (int j = 0; j < BK; ++j)
            if (j <= lim && j >= lo) mxs[j & 7] = fmaxf(mxs[j & 7], sv[j]);
        }
        const float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                               fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
        m2 = row_in ? mx * p.scale_log2 : 0.f;
        float ls[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) ls[j] = 0.f;
#pragma unroll
        for (int c = 0; c < BK / 32; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int ii = c * 32 + j;
            float p0 = ex2_approx(fmaf(sv[ii], p.scale_log2, -m2));
            float p1 = ex2_approx(fmaf(sv[ii + 1], p.scale_log2, -m2));
            if (!full) {
              p0 = (ii <= lim && ii >= lo) ? p0 : 0.f;
              p1 = (ii + 1 <= lim && ii + 1 >= lo) ? p1 : 0.f;
            }
            ls[(j >> 1) & 7] += p0 + p1;        // fp32 row sum (exact lse)
            pk[j / 2] = pack2<kFp16>(p0, p1);   // P rounded to 16 bits for the PV MMA
          }
          tmem_st16(tS + c * 16, pk);         // overwrites S columns already read
        }
        lsum = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&p_full[i & 1]);
      // the next tile's key range: its q_list read overlaps this epilogue
      const int2 nlr = nseq.valid() ? tile_lim(ndsc) : make_int2(-1, 0);

      // epilogue: O(i) -> 16-bit, one 64-column block at a time; each warp stages
      // its 32 rows in its own slots and TMA-stores them to the tile's
      // compact-buffer rows, so no warpgroup-wide barrier is needed
      mbar_wait_sticky(&o_full[i & 1], (i >> 1) & 1, p.status, &fail);
      tc_fence_after();
#pragma unroll
      for (int cb = 0; cb < kCB; ++cb) {
        uint32_t pk[32];
        {
          float ov[64];
          tmem_ld64(tO0 + os * D + cb * 64 + lane_off, ov);
#pragma unroll
          for (int j = 0; j < 64; j += 2) pk[j / 2] = pack2<kFp16>(ov[j], ov[j + 1]);
        }
        if (cb == kCB - 1) {
          tc_fence_before();
          mbar_arrive(&o_free[os]);
        }
        const uint32_t slot = stg + (n_cb % SS) * L::kStgW;
        // the slot's previous TMA store (this lane 0's bulk group) must have been read
        if (lane == 0 && n_cb >= SS) {
          if constexpr (SS == 2) bulk_wait_read_le1();
          else bulk_wait_read_all();
        }
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
          tma_store_2d_hint(&tm_o, slot, cb * 64, tile * kTileRows + (warp & 3) * 32, stream);
          bulk_commit();
        }
        ++n_cb;
      }
      st_global_v2_hint(p.mlbuf + (int64_t)tile * kTileRows + row, make_float2(m2, lsum), stream);
      seq = nseq;
      dsc = ndsc;
      lim = nlr.x;
      lo = nlr.y;
      nseq.next();
      nseq.next();
      ndsc = load_desc(p, nseq);
    }
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem_base, L::kTmemCols);
}

// Partial rows each lane keeps in flight in the merge.
#ifndef NSA_MERGE_BATCH
#define NSA_MERGE_BATCH 16
#endif

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
    const int32_t pr = p.prow[((int64_t)h * p.n + t) * p.topk + lane];
    if (pr >= 0) row = (int64_t)pr + j;
  }
  // The weights come first (the (m, l) loads and their reductions), then the partial
  // rows, kBatch at a time: with no loaded rows held across the reductions the kernel
  // needs 32 registers, so twice as many warps keep loads in flight as when the rows
  // were loaded first.
  constexpr int kBatch = NSA_MERGE_BATCH;
  const uint16_t *obuf = static_cast<const uint16_t *>(p.obuf);
  auto load_rows = [&](int k0, uint32_t (&u)[kBatch][E / 2]) {
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int64_t r = __shfl_sync(0xffffffffu, row, (k0 + b) & 31);
      const bool ok = k0 + b < p.topk && r >= 0;
      const uint16_t *src = obuf + (ok ? r : 0) * D + lane * E;
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
  };
  uint32_t u[kBatch][E / 2];
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
  for (int k0 = 0; k0 < p.topk; k0 += kBatch) {
    load_rows(k0, u);
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const float wk = __shfl_sync(0xffffffffu, w, (k0 + b) & 31);   // 0 for empty slots
#pragma unroll
      for (int e = 0; e < E / 2; ++e) {
        const float2 f = unpack2<kFp16>(u[b][e]);
        acc[2 * e] = fmaf(wk, f.x, acc[2 * e]);
        acc[2 * e + 1] = fmaf(wk, f.y, acc[2 * e + 1]);
      }
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

// Tensor map of a tile-padded compact buffer (forward partial O, backward partial
// dQ): [max_tiles * 128 rows, d], box = 32 rows x 64 columns (one warp's rows),
// 128-byte swizzle (the staging layout).
bool make_rows_map(const Params &p, void *base, int64_t max_tiles, CUtensorMap *m) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.d),
                              static_cast<cuuint64_t>(max_tiles) * kTileRows};
  const cuuint64_t str[1] = {static_cast<cuuint64_t>(p.d) * 2};
  const cuuint32_t box[2] = {64, 32};
  return encode_map(m, p.dtype == NSA_FP16, 2, base, dims, str, box);
}

// Tensor maps of k and v alone (the backward gathers q and dO with cp.async).
bool make_kv_maps(const Params &p, CUtensorMap *mk, CUtensorMap *mv) {
  const bool f16 = p.dtype == NSA_FP16;
  const cuuint64_t kdims[3] = {static_cast<cuuint64_t>(p.d), static_cast<cuuint64_t>(p.h_k),
                               static_cast<cuuint64_t>(p.n)};
  const cuuint64_t kstr[2] = {static_cast<cuuint64_t>(p.d) * 2,
                              static_cast<cuuint64_t>(p.h_k) * p.d * 2};
  const cuuint32_t kbox[3] = {64, 1, static_cast<cuuint32_t>(p.block)};
  return encode_map(mk, f16, 3, p.k, kdims, kstr, kbox) &&
         encode_map(mv, f16, 3, p.v, kdims, kstr, kbox);
}

template <int D, int BK, bool kFp16>
static cudaError_t run_fwd(const Params &p, int num_sms, int64_t max_tiles, cudaStream_t stream,
                           void (*mark)(int, cudaStream_t, bool)) {
  using L = FwdSmem<D, BK>;
  CUtensorMap mq, mk, mv, mo;
  if (!make_qkv_maps(p, p.q, &mq, &mk, &mv) || !make_rows_map(p, p.obuf, max_tiles, &mo))
    return cudaErrorInvalidValue;
  // One CTA per SM: it owns all 512 TMEM columns.
  const uint32_t smem = L::kBytes > 120u * 1024u ? L::kBytes : 120u * 1024u;
  auto kern = p.window > 0 ? fwd_main_kernel<D, BK, kFp16, true>
                            : fwd_main_kernel<D, BK, kFp16, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  int64_t grid = num_sms;
  if (grid > max_tiles) grid = max_tiles > 0 ? max_tiles : 1;
  mark(5, stream, true);
  kern<<<static_cast<unsigned>(grid), kFwdThreads, smem, stream>>>(mq, mk, mv, mo, p);
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
