// common.cuh -- shared definitions of the sm_103a selected-attention kernels:
// parameter blocks, workspace layout and thin inline-PTX wrappers for the
// Blackwell primitives used (tcgen05 MMA / TMEM, mbarrier, cp.async).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nsa_sel_attn.h"

namespace nsa {

// ---------------------------------------------------------------------------
// Tiling constants
// ---------------------------------------------------------------------------
constexpr int kTileRows = 128;      // gathered (token, query head) rows per MMA tile (tcgen05 M)
constexpr int kIdxThreads = 256;    // index builder: threads per CTA (one token per thread)
constexpr int kThreads = 128;       // backward main kernel: one thread per tile row / TMEM lane
constexpr int kScanPer = 4096;      // entries per CTA of the multi-CTA exclusive scan
constexpr int kMaxBwdCtas = 1024;   // backward main kernel: upper bound on its grid

// ---------------------------------------------------------------------------
// Workspace layout (byte offsets from the workspace base, all 256-aligned)
// ---------------------------------------------------------------------------
struct Layout {
  int64_t nb_max;          // upper bound on blocks per head: ceil(N/B_K) + S
  int64_t max_pairs;       // upper bound on kept (token, slot) pairs: h_k * N * T
  int64_t max_rows;        // max_pairs * g
  int64_t max_tiles;       // upper bound on 128-row tiles over the (head, block) segments
  int idx_tok;             // tokens per index-builder CTA (256, 128, 64 or 32)
  int64_t n_idx_tiles;     // token tiles of the index builder
  int n_w;                 // forward waves (token windows processed one after another)
  int wave_tiles;          // index token tiles per forward wave
  int64_t nsub;            // forward sub-segments: h_k * n_w * nb_max (head, wave, block)
  int64_t max_wtiles;      // upper bound on forward tiles over the sub-segments
  int64_t n_scan_ctas;     // CTAs of the sub-segment tile scan
  // index region
  size_t status, nb, blk_start, counts, offsets, tile_off, q_list, slot_map,
      chunk_hist, npairs, prow, wtile_off, wscan_part, tdesc, tseg;
  size_t index_end;
  // forward scratch
  size_t obuf, mlbuf;
  size_t fwd_end;
  // backward scratch
  size_t dstat, part_off, dqbuf, dkvbuf;
  int64_t max_parts;       // upper bound on backward dK/dV partial slots
  size_t bwd_end;
};

// Forward tile descriptor (one per 128-row tile of a (head, wave, block) sub-segment).
//   q_off : q_list index of the sub-segment's first token
//   row0  : first row of the tile inside the sub-segment (rows = token-major, g heads)
//   key0  : global index of the block's first key
//   hn    : KV head | (rows in this tile) << 16
struct TileDesc {
  int32_t q_off, row0, key0, hn;
};

// ---------------------------------------------------------------------------
// Kernel parameter block (shared by all kernels; plain pointers + sizes)
// ---------------------------------------------------------------------------
struct Params {
  // problem
  int32_t num_seqs, n, h_q, h_k, g, d, block, topk, dtype;
  float scale, scale_log2;
  // inputs
  const void *q, *k, *v, *out_in, *dout;
  const float *lse_in;
  const int32_t *sel, *cu;
  // outputs
  void *out, *dq, *dk, *dv;
  float *lse;
  // workspace views
  int32_t *status, *nb, *blk_start, *counts, *offsets, *tile_off, *q_list,
      *slot_map, *chunk_hist, *npairs, *prow, *wtile_off, *wscan_part;
  TileDesc *tdesc;
  int32_t *tseg;    // (head, block) segment of every forward tile
  int64_t nb_max, n_idx_tiles, nsub, n_scan_ctas;
  int idx_tok, n_w, wave_tiles;
  int fwd_chunk;    // forward schedule: consecutive tiles per chunk, chunks dealt round-robin
  int bwd_chunk;    // the same for the backward main kernel
  int window;       // sliding window: a row of token t sees keys >= t - window + 1 (0: none)
  void *obuf;       // forward partial outputs [tiles * 128, d] (dtype), tile-padded rows
  float2 *mlbuf;    // forward partial (max, sum) per padded row, log2 domain
  float *dstat;     // backward D = rowsum(dO * O) [h_q, N]
  int32_t *part_off;  // backward: first dK/dV partial slot of each segment [h_k * nb + 1]
  void *dqbuf;      // backward partial dQ [tiles * 128, d] (dtype), tile-padded rows
  float *dkvbuf;    // backward dK, dV partials [slots, 2, B_K, d] fp32
};

// ---------------------------------------------------------------------------
// Driver API entry points, resolved through the runtime at first use so that the
// library does not link libcuda and loads on a machine without a GPU driver.
// Returns nullptr when the driver (or the symbol) is missing.
// ---------------------------------------------------------------------------
template <typename Fn>
inline Fn driver_entry(const char *name) {
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(fn);
}

// ---------------------------------------------------------------------------
// Small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void set_status(int32_t *status, int32_t bits) {
  atomicOr(reinterpret_cast<int *>(status), bits);
}

// Largest s in [0, S) with cu[s] <= t (cu non-decreasing).
__device__ __forceinline__ int seq_of(const int32_t *cu, int num_seqs, int t) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Largest i in [0, n) with a[i] <= x (a non-decreasing, a[0] <= x).
__device__ __forceinline__ int upper_index(const int32_t *a, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier (bounded waits: give up after ~2 s and report NSA_DEVERR_TIMEOUT)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe of a phase (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Returns false (and flags the status word) when the phase did not complete in time.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int32_t *status) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(addr, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      set_status(status, NSA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Waits used by warp-specialised kernels: once any wait of the CTA has timed out
// (*fail set), every later wait returns at once, so all roles run their loops to
// the end with unchanged control flow (no thread is left behind at a barrier).
__device__ __forceinline__ bool mbar_wait_sticky(uint64_t *bar, uint32_t parity,
                                                 int32_t *status, volatile int *fail) {
  const uint32_t addr = smem_u32(bar);
  if (mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (*fail) return false;
    if (mbar_try_wait(addr, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *fail = 1;
      set_status(status, NSA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// ---------------------------------------------------------------------------
// TMA (tensor-map loads into 128-byte-swizzled tiles) and bulk stores
// ---------------------------------------------------------------------------
// 3-D tiled load; completion is counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap *map, int c0,
                                                 int c1, int c2, uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
      "l"(pol)
      : "memory");
}

// Four rows (r0..r3) of a 2-D tensor map with a one-row box, columns [col, col + box).
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *map, int col, int r0,
                                            int r1, int r2, int r3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_store(void *gdst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(src), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Named barrier; the non-aligned form, so lanes that reach it from different
// branches of the same warp are allowed.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// cp.async (16-byte global -> shared copies; src_bytes = 0 zero-fills)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// L2 eviction policies (createpolicy) for streaming stores and reused loads.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void *src, uint32_t src_bytes,
                                                uint64_t pol) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(dst),
               "l"(src), "r"(src_bytes), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_global_v2_hint(float2 *dst, float2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(dst), "f"(v.x),
               "f"(v.y), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// Wait until at most N of this thread's committed cp.async groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Generic-proxy shared-memory writes -> visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Shared-memory tiles in the 128-byte-swizzled layout used by tcgen05 operands.
// A tile of R rows x C 16-bit columns is stored as C/64 "column blocks"; column
// block cb holds, for each row r, 128 bytes (64 elements) at cb*R*128 + r*128,
// with its eight 16-byte chunks permuted chunk -> chunk ^ (r % 8).  Tile bases are
// 1024-byte aligned.  The same storage serves as a K-major operand (rows = M or N,
// columns = K) or as an MN-major operand (rows = K, columns = M or N).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk, int rows) {
  // chunk = 16-byte chunk index along the full row (8 chunks per column block)
  return static_cast<uint32_t>((chunk >> 3) * rows * 128 + row * 128 +
                               (((chunk & 7) ^ (row & 7)) << 4));
}

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle, sm_100 family version.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t desc = 0;
  desc |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  desc |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  desc |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  desc |= static_cast<uint64_t>(1) << 46;   // descriptor version (tcgen05)
  desc |= static_cast<uint64_t>(2) << 61;   // 128-byte swizzle
  return desc;
}

// K-major operand: rows are the M (or N) dimension, columns the K dimension.
// k-step s covers columns [16 s, 16 s + 16).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int rows, int s) {
  return sdesc_sw128(tile + (s >> 2) * rows * 128 + (s & 3) * 32, 16, 1024);
}

// MN-major operand: rows are the K dimension, columns the M (or N) dimension.
// k-step s covers rows [16 s, 16 s + 16); the next 64 M/N columns are one column
// block (rows * 128 bytes) further.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int rows, int s) {
  return sdesc_sw128(tile + s * 2048, rows * 128, 1024);
}

// The same descriptors split into their two 32-bit words, for kernels that keep
// the constant upper word and the stage base of the lower word in registers and
// step through k by adding to the 14-bit address field (addresses < 256 KB, so
// the field never carries into the leading-byte-offset field).
__host__ __device__ constexpr uint32_t sdesc_hi_sw128(uint32_t sbo) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (2u << 29);
}
__device__ __forceinline__ uint32_t sdesc_lo_sw128(uint32_t saddr, uint32_t lbo) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__device__ __forceinline__ uint64_t sdesc_join(uint32_t lo, uint32_t hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
  return d;
}
// Byte offset of k-step s inside a K-major (rows x K) 128-byte-swizzled tile,
// and inside an MN-major (K rows) tile, as used by desc_kmajor / desc_mnmajor.
__host__ __device__ constexpr uint32_t kmajor_step(int rows, int s) {
  return static_cast<uint32_t>((s >> 2) * rows * 128 + (s & 3) * 32);
}
__host__ __device__ constexpr uint32_t mnmajor_step(int s) { return static_cast<uint32_t>(s * 2048); }

// Instruction descriptor, kind::f16: D = f32, A/B = bf16 (or f16), dense.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n, bool a_mn, bool b_mn, bool fp16) {
  return (1u << 4) | ((fp16 ? 0u : 1u) << 7) | ((fp16 ? 0u : 1u) << 10) |
         ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  __syncwarp();
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  __syncwarp();
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T  (one elected thread issues)
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T: A is M x K with row m in TMEM lane m and two
// 16-bit K elements per 32-bit column (element k of the row in column k / 2, low
// half for even k).  Used for O += P V with P written to TMEM by the softmax.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once all previously issued tcgen05.mma of this thread complete.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// tcgen05.ld / tcgen05.st / tcgen05.wait are .sync.aligned: every lane of the warp
// must execute them together.  Inline asm hides that from the compiler, so each
// wrapper first reconverges the warp (its callers may come from data-dependent
// branches, e.g. the causal mask).
// 32 consecutive fp32 TMEM columns of this thread's lane, waited on before returning.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  __syncwarp();
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 64 consecutive fp32 TMEM columns of this thread's lane, one wait for all.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
  __syncwarp();
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
      "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 consecutive 32-bit TMEM columns of this thread's lane (a warp writes its
// 32-lane subpartition); the caller waits with tmem_wait_st before signalling.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  __syncwarp();
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  __syncwarp();
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2-D tiled TMA store from a 128-byte-swizzled shared-memory box (bulk group).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int c0,
                                             int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(src)
      : "memory");
}
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap *map, uint32_t src, int c0,
                                                  int c1, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint"
      " [%0, {%1, %2}], [%3], %4;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(src), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void bulk_wait_read_le1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The tiles of one CTA: chunks of `C` consecutive tiles, chunk c going to CTA
// c % gridDim.x.  C = 0 means one contiguous range per CTA.
struct TileSeq {
  int total, C, chunk, in_chunk;
  __device__ __forceinline__ void init(int total_, int c) {
    total = total_;
    C = c > 0 ? c : max(1, (total_ + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x));
    chunk = blockIdx.x;
    in_chunk = 0;
  }
  __device__ __forceinline__ int tile() const { return chunk * C + in_chunk; }
  __device__ __forceinline__ bool valid() const { return chunk * C + in_chunk < total; }
  __device__ __forceinline__ void next() {
    if (++in_chunk == C || chunk * C + in_chunk >= total) {
      in_chunk = 0;
      chunk += gridDim.x;
    }
  }
};

__device__ __forceinline__ TileDesc load_desc(const Params &p, const TileSeq &s) {
  if (!s.valid()) return TileDesc{0, 0, -1, -1};
  const int4 v = __ldg(reinterpret_cast<const int4 *>(p.tdesc) + s.tile());
  return TileDesc{v.x, v.y, v.z, v.w};
}

// ---------------------------------------------------------------------------
// Walks the 128-row tiles of consecutive (KV head, block) segments in order.
// set(t) moves to tile t (>= the previous one); `jseg` counts the distinct
// segments visited so far (0 for the first), which indexes K/V buffer slots.
// ---------------------------------------------------------------------------
struct TileCursor {
  int nb, nseg;
  int seg, seg_first_tile, seg_end_tile;
  int h, gb, key0, seg_off, seg_rows;
  int row0, nrows, jseg;
  bool new_seg;

  __device__ __forceinline__ void load_seg(const Params &p) {
    h = seg / nb;
    gb = seg - h * nb;
    const int s = upper_index(p.blk_start, p.num_seqs + 1, gb);
    key0 = p.cu[s] + (gb - p.blk_start[s]) * p.block;
    seg_off = p.offsets[seg];
    seg_rows = (p.offsets[seg + 1] - seg_off) * p.g;
    seg_first_tile = p.tile_off[seg];
    seg_end_tile = p.tile_off[seg + 1];
  }
  __device__ __forceinline__ void start(const Params &p, int nb_, int tile0) {
    nb = nb_;
    nseg = p.h_k * nb_;
    seg = upper_index(p.tile_off, nseg + 1, tile0);
    load_seg(p);
    jseg = -1;
    new_seg = true;
  }
  // Tile `t` must be >= every tile passed before; the first call starts segment 0.
  __device__ __forceinline__ void set(const Params &p, int t) {
    bool moved = jseg < 0;
    if (t >= seg_end_tile) {
      while (p.tile_off[seg + 1] <= t) ++seg;
      load_seg(p);
      moved = true;
    }
    new_seg = moved;
    if (moved) ++jseg;
    row0 = (t - seg_first_tile) * 128;
    nrows = min(128, seg_rows - row0);
  }
};

// ---------------------------------------------------------------------------
// dtype helpers (bf16 / fp16 stored as raw 16-bit)
// ---------------------------------------------------------------------------
template <bool kFp16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (kFp16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}
template <bool kFp16>
__device__ __forceinline__ float2 unpack2(uint32_t u) {
  if constexpr (kFp16) {
    __half2 h = *reinterpret_cast<__half2 *>(&u);
    return __half22float2(h);
  } else {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(h);
  }
}
template <bool kFp16>
__device__ __forceinline__ float round16(float x) {
  if constexpr (kFp16) return __half2float(__float2half_rn(x));
  else return __bfloat162float(__float2bfloat16_rn(x));
}

}  // namespace nsa
