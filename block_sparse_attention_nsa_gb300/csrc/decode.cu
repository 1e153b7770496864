// decode.cu -- one-step decode of NSA selected attention on sm_103a.
//
// The one-step decoding preview of the Flash-Sparse-Attention README ("News") and
// the decoding stage that "FSA: An Alternative Efficient Implementation of Native
// Sparse Attention Kernel" leaves open (局限与展望): each sequence has one new query
// token, the last token of its KV cache, and it attends to the keys of the blocks its
// selection names -- the same arithmetic as the forward for that token (causal mask,
// one softmax over the union of the kept blocks).
//
// Per (sequence, KV head) the work is T blocks of K and V read once and 4 d g B_K T
// FLOP on them, with g <= 16 query rows: HBM-bound, far too few rows for a tensor-core
// tile, so CUDA cores do it.  One CTA of 8 warps per (sequence, KV head); warp w takes
// kept blocks w, w + 8, ... in sub-blocks of 32 keys:
//   K rows are staged by cp.async in padded shared-memory rows, the next sub-block's
//   while this one is computed; lane l owns key l of a 32-key sub-block: S = q K^T for
//   the g heads (q, pre-scaled by scale * log2 e, read from shared memory as a
//   broadcast); online softmax per head; P to shared memory; O += P V with V rows read
//   straight from global memory, eight rows in flight ahead, lane l owning d elements
//   [E l, E l + E).  The warps' (m, l, O) are merged in shared memory at the
//   end: out and lse are written once, no workspace.
#include "common.cuh"

namespace nsa {

constexpr int kDecWarps = 8;
constexpr int kDecMaxG = 16;

struct DecodeParams {
  int num_seqs, h_q, h_k, g, block, topk;
  float scale_log2;
  const void *q;          // [B, h_q, d]
  const void *k, *v;      // [N, h_k, d]
  const int32_t *sel;     // [h_k, B, T]
  const int32_t *cu;      // [B + 1]
  void *out;              // [B, h_q, d]
  float *lse;             // [h_q, B]
  int32_t *status;        // device status word (may be null)
};

template <int D, int GM>
struct DecSmem {
  static constexpr int KS = 32;                        // keys per sub-block (one per lane)
  static constexpr uint32_t kRow = D * 2 + 16;         // padded K row (bytes)
  static constexpr uint32_t kStage = KS * kRow;        // one K sub-block
  static constexpr uint32_t kOffQ = 0;                 // q, fp32 [GM][D]
  static constexpr uint32_t kOffP = kOffQ + GM * D * 4;    // P, fp32 [warp][GM][KS]
  static constexpr uint32_t kOffK = kOffP + kDecWarps * GM * KS * 4;   // [warp][2][stage]
  static constexpr uint32_t kOffL = kOffK + kDecWarps * 2 * kStage;   // kept blocks [32]
  static constexpr uint32_t kBytes = kOffL + 32 * 4 + 16;
  // the merge area [warp][GM][D + 2] reuses the K staging
  static_assert(kDecWarps * GM * (D + 2) * 4 <= kDecWarps * 2 * kStage, "merge area");
};

// Two CTAs per SM when the per-head state is small (g <= 4), one otherwise.
template <int D, int BK, int GM, bool kFp16>
__global__ void __launch_bounds__(kDecWarps * 32, GM <= 4 ? 2 : 1) decode_kernel(DecodeParams p) {
  using L = DecSmem<D, GM>;
  constexpr int KS = L::KS;               // keys per sub-block: lane l owns key l
  constexpr int NK = KS / 32;
  constexpr int E = D / 32;               // d elements per lane in O
  constexpr int kCPR = D / 8;             // 16-byte chunks per row
  extern __shared__ __align__(16) uint8_t smem[];
  float *qs = reinterpret_cast<float *>(smem + L::kOffQ);
  int32_t *kept = reinterpret_cast<int32_t *>(smem + L::kOffL);
  __shared__ int n_kept;
  const int b = blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = p.g;
  const int t0 = p.cu[b], len = p.cu[b + 1] - t0;
  const int nblk = len > 0 ? (len + BK - 1) / BK : 0;
  const int c = len > 0 ? (len - 1) / BK : -1;   // the query token's own block

  // q of the g heads, fp32, pre-scaled by scale * log2 e
  const uint16_t *gq = static_cast<const uint16_t *>(p.q) + ((int64_t)b * p.h_q + h * g) * D;
  for (int i = tid; i < g * D; i += blockDim.x) {
    const uint32_t two = gq[i];
    qs[i] = (kFp16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(two)))
                   : __uint_as_float(two << 16)) * p.scale_log2;
  }
  // the kept blocks: valid, causal, first occurrence of each value
  if (warp == 0) {
    const int32_t *row = p.sel + ((int64_t)h * p.num_seqs + b) * p.topk;
    const int blk = lane < p.topk ? row[lane] : -1;
    bool bad = lane < p.topk && (blk < -1 || blk >= nblk);
    bool ok = lane < p.topk && blk >= 0 && blk <= c;
#pragma unroll 1
    for (int j = 0; j < 32; ++j) {
      const int other = __shfl_sync(0xffffffffu, blk, j);
      if (j < lane && other == blk) ok = false;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, ok);
    if (ok) kept[__popc(m & ((1u << lane) - 1u))] = blk;
    if (lane == 0) n_kept = __popc(m);
    if (__any_sync(0xffffffffu, bad) && lane == 0 && p.status)
      atomicOr(p.status, NSA_DEVERR_BAD_INDEX);
  }
  __syncthreads();
  const int nk = n_kept;

  float m_run[GM], l_run[GM], o[GM][E];
#pragma unroll
  for (int hh = 0; hh < GM; ++hh) {
    m_run[hh] = -INFINITY;
    l_run[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[hh][e] = 0.f;
  }
  const uint32_t stage0 = smem_u32(smem + L::kOffK + warp * 2 * L::kStage);
  float *pw = reinterpret_cast<float *>(smem + L::kOffP) + warp * GM * KS;
  const uint16_t *gk = static_cast<const uint16_t *>(p.k);
  const uint16_t *gv = static_cast<const uint16_t *>(p.v);
  const int64_t rstride = (int64_t)p.h_k * D;   // elements between consecutive tokens
  // This warp's sub-blocks: n = 0, 1, ... -> kept block w + 8 (n / SPB), part n % SPB.
  constexpr int SPB = BK / KS;
  const int nmine = nk > warp ? ((nk - 1 - warp) / kDecWarps + 1) * SPB : 0;
  auto sub_key0 = [&](int n) { return kept[warp + kDecWarps * (n / SPB)] * BK + (n % SPB) * KS; };
  // K rows of sub-block n into buffer n % 2 (zero-filled past the sequence end)
  auto stage_k = [&](int n) {
    const int key0 = sub_key0(n), nkeys = min(KS, len - key0);
    const uint32_t st = stage0 + (n & 1) * L::kStage;
    const uint16_t *kbase = gk + ((int64_t)(t0 + key0)) * rstride + (int64_t)h * D;
#pragma unroll 4
    for (int i = lane; i < KS * kCPR; i += 32) {
      const int r = i / kCPR, ch = i % kCPR;
      const bool in = r < nkeys;
      cp_async16(st + r * L::kRow + ch * 16, kbase + (in ? (int64_t)r * rstride + ch * 8 : 0),
                 in ? 16u : 0u);
    }
    cp_async_commit();
  };
  if (nmine > 0) stage_k(0);
  for (int n = 0; n < nmine; ++n) {
    const int key0 = sub_key0(n);
    const int nkeys = min(KS, len - key0);           // keys of this sub-block that exist
    if (nkeys <= 0) {                                 // past the sequence end: nothing here
      cp_async_wait_all();
      __syncwarp();
      if (n + 1 < nmine) stage_k(n + 1);
      continue;
    }
    // the next sub-block's K is in flight while this one is computed
    if (n + 1 < nmine) {
      stage_k(n + 1);
      cp_async_wait_group<1>();
    } else {
      cp_async_wait_all();
    }
    __syncwarp();
    const uint32_t stage = stage0 + (n & 1) * L::kStage;
    // the first V rows of this sub-block are loaded now, to land during S
    const uint16_t *vbase = gv + ((int64_t)(t0 + key0)) * rstride + (int64_t)h * D + lane * E;
    auto load_v = [&](int k0, uint32_t (&w)[8][E / 2]) {
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const bool in = k0 + u < nkeys;
        const uint16_t *src = vbase + (in ? (int64_t)(k0 + u) * rstride : 0);
        if constexpr (E == 2) {
          w[u][0] = in ? __ldg(reinterpret_cast<const unsigned int *>(src)) : 0u;
        } else if constexpr (E == 4) {
          const uint2 x = in ? __ldg(reinterpret_cast<const uint2 *>(src)) : make_uint2(0u, 0u);
          w[u][0] = x.x; w[u][1] = x.y;
        } else {
          const uint4 x = in ? __ldg(reinterpret_cast<const uint4 *>(src))
                             : make_uint4(0u, 0u, 0u, 0u);
          w[u][0] = x.x; w[u][1] = x.y; w[u][2] = x.z; w[u][3] = x.w;
        }
      }
    };
    uint32_t vw[8][E / 2];
    load_v(0, vw);
    // ---- S for the lane's key, all heads ----
    float s[GM][NK];
#pragma unroll
    for (int hh = 0; hh < GM; ++hh)
#pragma unroll
      for (int i = 0; i < NK; ++i) s[hh][i] = 0.f;
#pragma unroll 2
    for (int ch = 0; ch < kCPR; ++ch) {
      float kf[NK][8];
#pragma unroll
      for (int i = 0; i < NK; ++i) {
        uint4 raw;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(raw.x), "=r"(raw.y), "=r"(raw.z), "=r"(raw.w)
                     : "r"(stage + (lane + 32 * i) * L::kRow + ch * 16));
        const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 f = unpack2<kFp16>(w4[u]);
          kf[i][2 * u] = f.x;
          kf[i][2 * u + 1] = f.y;
        }
      }
#pragma unroll
      for (int hh = 0; hh < GM; ++hh) {
        if (hh < g) {
          const float4 qa = *reinterpret_cast<const float4 *>(qs + hh * D + ch * 8);
          const float4 qb = *reinterpret_cast<const float4 *>(qs + hh * D + ch * 8 + 4);
#pragma unroll
          for (int i = 0; i < NK; ++i) {
            float a = s[hh][i];
            a = fmaf(qa.x, kf[i][0], a); a = fmaf(qa.y, kf[i][1], a);
            a = fmaf(qa.z, kf[i][2], a); a = fmaf(qa.w, kf[i][3], a);
            a = fmaf(qb.x, kf[i][4], a); a = fmaf(qb.y, kf[i][5], a);
            a = fmaf(qb.z, kf[i][6], a); a = fmaf(qb.w, kf[i][7], a);
            s[hh][i] = a;
          }
        }
      }
    }
    // ---- online softmax per head; P to shared memory ----
#pragma unroll
    for (int hh = 0; hh < GM; ++hh) {
      if (hh < g) {
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < NK; ++i)
          if (lane + 32 * i < nkeys) mx = fmaxf(mx, s[hh][i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m_run[hh], mx);
        const float alpha = ex2_approx(m_run[hh] - m_new);   // 0 on the first sub-block
        float ps = 0.f;
#pragma unroll
        for (int i = 0; i < NK; ++i) {
          const float pv = (lane + 32 * i < nkeys) ? ex2_approx(s[hh][i] - m_new) : 0.f;
          pw[hh * KS + lane + 32 * i] = pv;
          ps += pv;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        l_run[hh] = l_run[hh] * alpha + ps;
        m_run[hh] = m_new;
#pragma unroll
        for (int e = 0; e < E; ++e) o[hh][e] *= alpha;
      }
    }
    __syncwarp();
    // ---- O += P V, eight V rows at a time, the next eight in flight ----
#pragma unroll 1
    for (int k0 = 0; k0 < nkeys; k0 += 8) {
      float vf[8][E];
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int e = 0; e < E / 2; ++e) {
          const float2 f = unpack2<kFp16>(vw[u][e]);
          vf[u][2 * e] = f.x;
          vf[u][2 * e + 1] = f.y;
        }
      if (k0 + 8 < nkeys) load_v(k0 + 8, vw);
#pragma unroll
      for (int hh = 0; hh < GM; ++hh) {
        if (hh < g) {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float pv = pw[hh * KS + k0 + u];   // 0 past nkeys
#pragma unroll
            for (int e = 0; e < E; ++e) o[hh][e] = fmaf(pv, vf[u][e], o[hh][e]);
          }
        }
      }
    }
    __syncwarp();   // P and this K buffer are rewritten two sub-blocks later
  }
  cp_async_wait_all();

  // ---- merge the warps' (m, l, O) per head ----
  __syncthreads();   // every warp is done with its K stage: the merge area reuses it
  float *mg = reinterpret_cast<float *>(smem + L::kOffK);   // [warp][GM][D + 2]
#pragma unroll
  for (int hh = 0; hh < GM; ++hh) {
    if (hh < g) {
      float *dst = mg + ((size_t)warp * GM + hh) * (D + 2);
#pragma unroll
      for (int e = 0; e < E; ++e) dst[lane * E + e] = o[hh][e];
      if (lane == 0) {
        dst[D] = m_run[hh];
        dst[D + 1] = l_run[hh];
      }
    }
  }
  __syncthreads();
  for (int hh = warp; hh < g; hh += kDecWarps) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, mg[((size_t)w * GM + hh) * (D + 2) + D]);
    float lsum = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
    for (int w = 0; w < kDecWarps; ++w) {
      const float *src = mg + ((size_t)w * GM + hh) * (D + 2);
      const float mw = src[D];
      const float wt = (mw == -INFINITY) ? 0.f : ex2_approx(mw - M);
      lsum += wt * src[D + 1];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(wt, src[lane * E + e], acc[e]);
    }
    const bool any = lsum > 0.f;
    const float inv = any ? 1.f / lsum : 0.f;
    uint16_t *dst = static_cast<uint16_t *>(p.out) + ((int64_t)b * p.h_q + h * g + hh) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2)
      *reinterpret_cast<uint32_t *>(dst + e) = pack2<kFp16>(acc[e] * inv, acc[e + 1] * inv);
    if (lane == 0)
      p.lse[(int64_t)(h * g + hh) * p.num_seqs + b] =
          any ? (M + __log2f(lsum)) * 0.69314718055994531f : -INFINITY;
  }
}

template <int D, int BK, int GM, bool kFp16>
static cudaError_t run_decode(const DecodeParams &p, cudaStream_t s) {
  using L = DecSmem<D, GM>;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, BK, GM, kFp16>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(L::kBytes));
  if (e != cudaSuccess) return e;
  decode_kernel<D, BK, GM, kFp16>
      <<<dim3(static_cast<unsigned>(p.num_seqs), static_cast<unsigned>(p.h_k)), kDecWarps * 32,
         L::kBytes, s>>>(p);
  return cudaGetLastError();
}

template <int D, bool kFp16>
static cudaError_t run_decode_bk(const DecodeParams &p, cudaStream_t s) {
  const bool small = p.g <= 4;
  switch (p.block) {
    case 32: return small ? run_decode<D, 32, 4, kFp16>(p, s) : run_decode<D, 32, 16, kFp16>(p, s);
    case 64: return small ? run_decode<D, 64, 4, kFp16>(p, s) : run_decode<D, 64, 16, kFp16>(p, s);
    case 128:
      return small ? run_decode<D, 128, 4, kFp16>(p, s) : run_decode<D, 128, 16, kFp16>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode(int num_seqs, int h_q, int h_k, int d, int block, int topk, bool fp16,
                          float scale, const void *q, const void *k, const void *v,
                          const int32_t *sel, const int32_t *cu, void *out, float *lse,
                          int32_t *status, cudaStream_t s) {
  DecodeParams p;
  p.num_seqs = num_seqs;
  p.h_q = h_q;
  p.h_k = h_k;
  p.g = h_q / h_k;
  p.block = block;
  p.topk = topk;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q = q;
  p.k = k;
  p.v = v;
  p.sel = sel;
  p.cu = cu;
  p.out = out;
  p.lse = lse;
  p.status = status;
  if (p.g > kDecMaxG) return cudaErrorInvalidValue;
  switch (d) {
    case 64: return fp16 ? run_decode_bk<64, true>(p, s) : run_decode_bk<64, false>(p, s);
    case 128: return fp16 ? run_decode_bk<128, true>(p, s) : run_decode_bk<128, false>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nsa
