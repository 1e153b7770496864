// api.cu -- the C ABI (include/nsa_sel_attn.h): argument validation, workspace
// layout, kernel launches and the optional per-kernel event timing.
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "compress.cuh"

namespace nsa {
cudaError_t launch_index(const Params &p, cudaStream_t s, void (*mark)(int, cudaStream_t, bool));
cudaError_t index_set_smem_limits(const Params &p);
cudaError_t launch_fwd(const Params &p, int num_sms, int64_t max_tiles, cudaStream_t s,
                       void (*mark)(int, cudaStream_t, bool));
cudaError_t launch_window_select(const int32_t *cu, int num_seqs, int n, int h_k, int block,
                                 int topk, int window, int32_t *sel, cudaStream_t s);
cudaError_t launch_gate_combine(int64_t rows, int d, bool fp16, int nbr, const void *o0,
                                const void *o1, const void *o2, const float *gates, void *out,
                                const void *dout, void *d0, void *d1, void *d2, float *dgates,
                                bool bwd, cudaStream_t s);
cudaError_t launch_decode(int num_seqs, int h_q, int h_k, int d, int block, int topk, bool fp16,
                          float scale, const void *q, const void *k, const void *v,
                          const int32_t *sel, const int32_t *cu, void *out, float *lse,
                          int32_t *status, cudaStream_t s);
cudaError_t launch_bwd(const Params &p, int num_sms, int64_t max_tiles, cudaStream_t s,
                       void (*mark)(int, cudaStream_t, bool));
cudaError_t launch_cmp_offsets(const int32_t *cu, int num_seqs, int n, int ksize, int stride,
                               int32_t *cu_cmp, int32_t *status, cudaStream_t s);
cudaError_t launch_compress(int d, bool fp16, const int32_t *cu, const int32_t *cu_cmp,
                            int num_seqs, int n, int h_k, int ksize, int stride,
                            int64_t rows_cap, const void *k, const void *v, void *kc, void *vc,
                            cudaStream_t s);
cudaError_t launch_cmp_select(int d, bool fp16, const CmpParams &p, cudaStream_t s);
int cmp_tokens_per_cta(int d, int g, int nb_max, bool in_smem);

namespace {

constexpr int kNumKernels = 11;
const char *const kKernelNames[kNumKernels] = {
    "index_geometry", "index_count", "index_col_scan", "index_scans_and_tiles", "index_scatter",
    "fwd_main", "fwd_merge", "bwd_preprocess", "bwd_main", "bwd_dq_reduce", "bwd_dkv_reduce"};

// ---- per-kernel event timing (diagnostics; single host thread) ----
struct Rec {
  int id;
  cudaEvent_t a, b;
};
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> pool;
  std::vector<Rec> recs;
  size_t used = 0;
  cudaEvent_t pending = nullptr;
  int pending_id = -1;
  cudaEvent_t get() {
    if (used == pool.size()) {
      cudaEvent_t e;
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
      pool.push_back(e);
    }
    return pool[used++];
  }
} g_prof;

// Set by the host-buffer step around its backward: recorded once dk and dv are
// final (the end of the dK/dV reduction, kernel id 10).
thread_local cudaEvent_t t_dkv_ready = nullptr;
thread_local bool t_dkv_recorded = false;

void mark(int id, cudaStream_t stream, bool begin) {
  if (id == 10 && !begin && t_dkv_ready)
    t_dkv_recorded = cudaEventRecord(t_dkv_ready, stream) == cudaSuccess;
  if (!g_prof.on) return;
  cudaEvent_t e = g_prof.get();
  if (!e) return;
  cudaEventRecord(e, stream);
  if (begin) {
    g_prof.pending = e;
    g_prof.pending_id = id;
  } else if (g_prof.pending && g_prof.pending_id == id) {
    g_prof.recs.push_back({id, g_prof.pending, e});
    g_prof.pending = nullptr;
  }
}

int num_sms_cached() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 148;
  }
  return cache[dev];
}

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

nsa_status check_dims(const nsa_sel_attn_dims *d, bool bwd) {
  if (!d) return NSA_ERR_INVALID_ARG;
  if (d->num_seqs < 1 || d->total_tokens < 0 || d->h_k < 1 || d->h_q < 1 || d->topk < 1)
    return NSA_ERR_INVALID_ARG;
  if (d->h_q % d->h_k != 0) return NSA_ERR_INVALID_ARG;
  if (d->dtype != NSA_BF16 && d->dtype != NSA_FP16) return NSA_ERR_UNSUPPORTED;
  if (!(d->head_dim == 64 || d->head_dim == 128 || d->head_dim == 256)) return NSA_ERR_UNSUPPORTED;
  // backward with d = 256: B_K <= 64 (its shared memory holds one 64 KB Q/dO stage pair)
  if (bwd && d->head_dim == 256 && d->block_size > 64) return NSA_ERR_UNSUPPORTED;

  if (!(d->block_size == 32 || d->block_size == 64 || d->block_size == 128))
    return NSA_ERR_UNSUPPORTED;
  if (d->topk > 32) return NSA_ERR_UNSUPPORTED;
  const int64_t pairs = (int64_t)d->h_k * d->total_tokens * d->topk;
  const int64_t g = d->h_q / d->h_k;
  if (pairs >= (int64_t(1) << 31) || pairs * g >= (int64_t(1) << 31)) return NSA_ERR_UNSUPPORTED;
  if ((int64_t)d->total_tokens * d->h_q >= (int64_t(1) << 31)) return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

// Forward schedule: chunks of kFwdChunk consecutive tiles dealt round-robin to
// the CTAs, so that all CTAs work on neighbouring (head, block) segments at any
// time and the Q rows and K/V blocks they read stay L2-resident.
#ifndef NSA_FWD_CHUNK
#define NSA_FWD_CHUNK 4
#endif
constexpr int kFwdChunk = NSA_FWD_CHUNK;
// Backward schedule: the same dealing; the backward also writes one dK/dV partial per
// (segment, chunk) pair, so longer chunks mean fewer partials.  Chunk lengths measured
// on the 64K workload (forward 2/4/8/16, backward 8/16/32/64): 4 and 32 give the
// shortest forward + backward step at g = 4.
#ifndef NSA_BWD_CHUNK
#define NSA_BWD_CHUNK 32
#endif
constexpr int kBwdChunk = NSA_BWD_CHUNK;

// Shared memory the index builder may use per CTA (count: one int per block;
// scatter: one bit per (token, block) of the CTA's token tile).
constexpr int64_t kIdxSmemCap = 160 * 1024;

// Attention kernels not offered: d = 128 with B_K = 128, whose forward kernel raised
// an illegal-instruction fault on one ragged workload, cause not yet found.  The index
// builder and the workspace query do not depend on d and still accept it.
nsa_status check_kernels(const nsa_sel_attn_dims *d) {
  if (d->head_dim == 128 && d->block_size == 128) return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

nsa_status make_layout(const nsa_sel_attn_dims *d, Layout *L) {
  const int64_t N = d->total_tokens, B = d->block_size, S = d->num_seqs, T = d->topk;
  const int64_t g = d->h_q / d->h_k, h_k = d->h_k;
  L->nb_max = (N + B - 1) / B + S;
  L->max_pairs = h_k * N * T;
  L->max_rows = L->max_pairs * g;
  L->max_tiles = (L->max_rows + kTileRows - 1) / kTileRows + h_k * L->nb_max;
  if (L->nb_max * 4 > kIdxSmemCap) return NSA_ERR_UNSUPPORTED;
  // scatter: token masks (1 bit), warp prefixes (1 byte) and two bases per block
  auto scatter_bytes = [&](int tok) {
    return (tok / 32) * L->nb_max * 5 + 2 * L->nb_max * 4 + 16;
  };
  int tok = kIdxThreads;
  while (tok > 32 && scatter_bytes(tok) > kIdxSmemCap) tok >>= 1;
  if (scatter_bytes(tok) > kIdxSmemCap) return NSA_ERR_UNSUPPORTED;
  L->idx_tok = tok;
  L->n_idx_tiles = (N + tok - 1) / tok;
  if (L->n_idx_tiles < 1) L->n_idx_tiles = 1;
  // One wave over all tokens: sub-segments coincide with the (head, block) segments.
  L->wave_tiles = static_cast<int>(L->n_idx_tiles);
  L->n_w = 1;
  L->nsub = h_k * L->n_w * L->nb_max;
  L->max_wtiles = (L->max_rows + kTileRows - 1) / kTileRows + L->nsub;
  L->n_scan_ctas = (L->nsub + kScanPer - 1) / kScanPer;
  if (L->max_tiles >= (int64_t(1) << 31) / kTileRows ||
      L->max_wtiles >= (int64_t(1) << 31) / kTileRows)
    return NSA_ERR_UNSUPPORTED;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align256(o + bytes);
    return at;
  };
  const size_t nseg1 = static_cast<size_t>(h_k * L->nb_max + 1);
  const size_t hn = static_cast<size_t>(h_k * N > 0 ? h_k * N : 1);
  const size_t hnt = static_cast<size_t>(h_k * N * T > 0 ? h_k * N * T : 1);
  L->status = take(256);
  L->nb = take(4);
  L->blk_start = take(4 * static_cast<size_t>(S + 1));
  L->counts = take(4 * nseg1);
  L->offsets = take(4 * nseg1);
  L->tile_off = take(4 * nseg1);
  L->q_list = take(4 * static_cast<size_t>(L->max_pairs > 0 ? L->max_pairs : 1));
  L->slot_map = take(4 * hnt);
  L->chunk_hist = take(4 * static_cast<size_t>(h_k * L->n_idx_tiles * L->nb_max));
  L->npairs = take(4 * hn);
  L->prow = take(4 * hnt);
  L->wtile_off = take(4 * static_cast<size_t>(L->nsub + 1));
  L->wscan_part = take(4 * static_cast<size_t>(L->n_scan_ctas));
  L->tdesc = take(sizeof(TileDesc) * static_cast<size_t>(L->max_wtiles));
  L->tseg = take(4 * static_cast<size_t>(L->max_wtiles));
  L->index_end = o;
  const size_t scratch = o;
  L->obuf = take(static_cast<size_t>(L->max_wtiles) * kTileRows * d->head_dim * 2);
  L->mlbuf = take(static_cast<size_t>(L->max_wtiles) * kTileRows * 8);
  L->fwd_end = o;
  o = scratch;
  // backward: one dK/dV partial per (segment, chunk) pair a segment's tiles meet, at
  // most segments + chunk boundaries
  L->max_parts = h_k * L->nb_max + L->max_wtiles / kBwdChunk + 1;
  L->dstat = take(4 * static_cast<size_t>(N) * d->h_q);
  L->part_off = take(4 * nseg1);
  L->dqbuf = take(static_cast<size_t>(L->max_wtiles) * kTileRows * d->head_dim * 2);
  L->dkvbuf = take(static_cast<size_t>(L->max_parts) * 2 * B * d->head_dim * 4);
  L->bwd_end = o;
  return NSA_OK;
}

void fill_params(Params *p, const nsa_sel_attn_dims *d, const Layout &L, void *ws) {
  std::memset(p, 0, sizeof(*p));
  p->num_seqs = d->num_seqs;
  p->n = d->total_tokens;
  p->h_q = d->h_q;
  p->h_k = d->h_k;
  p->g = d->h_q / d->h_k;
  p->d = d->head_dim;
  p->block = d->block_size;
  p->topk = d->topk;
  p->dtype = d->dtype;
  char *w = static_cast<char *>(ws);
  p->status = reinterpret_cast<int32_t *>(w + L.status);
  p->nb = reinterpret_cast<int32_t *>(w + L.nb);
  p->blk_start = reinterpret_cast<int32_t *>(w + L.blk_start);
  p->counts = reinterpret_cast<int32_t *>(w + L.counts);
  p->offsets = reinterpret_cast<int32_t *>(w + L.offsets);
  p->tile_off = reinterpret_cast<int32_t *>(w + L.tile_off);
  p->q_list = reinterpret_cast<int32_t *>(w + L.q_list);
  p->slot_map = reinterpret_cast<int32_t *>(w + L.slot_map);
  p->chunk_hist = reinterpret_cast<int32_t *>(w + L.chunk_hist);
  p->npairs = reinterpret_cast<int32_t *>(w + L.npairs);
  p->prow = reinterpret_cast<int32_t *>(w + L.prow);
  p->wtile_off = reinterpret_cast<int32_t *>(w + L.wtile_off);
  p->wscan_part = reinterpret_cast<int32_t *>(w + L.wscan_part);
  p->tdesc = reinterpret_cast<TileDesc *>(w + L.tdesc);
  p->tseg = reinterpret_cast<int32_t *>(w + L.tseg);
  p->nb_max = L.nb_max;
  p->n_idx_tiles = L.n_idx_tiles;
  p->nsub = L.nsub;
  p->n_scan_ctas = L.n_scan_ctas;
  p->idx_tok = L.idx_tok;
  p->n_w = L.n_w;
  p->wave_tiles = L.wave_tiles;
  p->fwd_chunk = kFwdChunk;
  p->bwd_chunk = kBwdChunk;
  p->obuf = w + L.obuf;
  p->mlbuf = reinterpret_cast<float2 *>(w + L.mlbuf);
  p->dstat = reinterpret_cast<float *>(w + L.dstat);
  p->part_off = reinterpret_cast<int32_t *>(w + L.part_off);
  p->dqbuf = w + L.dqbuf;
  p->dkvbuf = reinterpret_cast<float *>(w + L.dkvbuf);
}

nsa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NSA_OK : NSA_ERR_CUDA; }

nsa_status run_index(const nsa_sel_attn_dims *d, const Layout &L, Params &p, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(p.status, 0, 4, s);
  if (e != cudaSuccess) return NSA_ERR_CUDA;
  e = index_set_smem_limits(p);
  if (e != cudaSuccess) return NSA_ERR_CUDA;
  (void)d;
  return cuda_status(launch_index(p, s, mark));
}

}  // namespace
}  // namespace nsa

using namespace nsa;

extern "C" {

nsa_status nsa_sel_attn_workspace_size(const nsa_sel_attn_dims *dims, size_t *fwd_bytes,
                                       size_t *bwd_bytes) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  Layout L;
  st = make_layout(dims, &L);
  if (st != NSA_OK) return st;
  if (fwd_bytes) *fwd_bytes = L.fwd_end;
  if (bwd_bytes) *bwd_bytes = L.bwd_end;
  return NSA_OK;
}

nsa_status nsa_sel_attn_index(const nsa_sel_attn_dims *dims, const int32_t *sel_idx,
                              const int32_t *cu_seqlens, void *workspace, size_t workspace_bytes,
                              nsa_stream_t stream) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  if (!cu_seqlens || !workspace || (dims->total_tokens > 0 && !sel_idx)) return NSA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return NSA_ERR_INVALID_ARG;
  Layout L;
  st = make_layout(dims, &L);
  if (st != NSA_OK) return st;
  if (workspace_bytes < L.index_end) return NSA_ERR_WORKSPACE;
  Params p;
  fill_params(&p, dims, L, workspace);
  p.sel = sel_idx;
  p.cu = cu_seqlens;
  return run_index(dims, L, p, reinterpret_cast<cudaStream_t>(stream));
}

nsa_status nsa_sel_attn_index_view(const nsa_sel_attn_dims *dims, const void *workspace,
                                   const int32_t **counts, const int32_t **offsets,
                                   const int32_t **q_list, const int32_t **slot_map,
                                   const int32_t **nb_device, int32_t *num_blocks) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  if (!workspace) return NSA_ERR_INVALID_ARG;
  Layout L;
  st = make_layout(dims, &L);
  if (st != NSA_OK) return st;
  const char *w = static_cast<const char *>(workspace);
  if (counts) *counts = reinterpret_cast<const int32_t *>(w + L.counts);
  if (offsets) *offsets = reinterpret_cast<const int32_t *>(w + L.offsets);
  if (q_list) *q_list = reinterpret_cast<const int32_t *>(w + L.q_list);
  if (slot_map) *slot_map = reinterpret_cast<const int32_t *>(w + L.slot_map);
  if (nb_device) *nb_device = reinterpret_cast<const int32_t *>(w + L.nb);
  if (num_blocks) *num_blocks = static_cast<int32_t>(L.nb_max);
  return NSA_OK;
}

static nsa_status fwd_impl(const nsa_sel_attn_dims *dims, const void *q, const void *k,
                           const void *v, const int32_t *sel_idx, const int32_t *cu_seqlens,
                           float scale, int window, void *out, float *lse, void *workspace,
                           size_t workspace_bytes, nsa_stream_t stream) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  st = check_kernels(dims);
  if (st != NSA_OK) return st;
  if (!cu_seqlens || !workspace || !std::isfinite(scale)) return NSA_ERR_INVALID_ARG;
  if (dims->total_tokens > 0 && (!q || !k || !v || !sel_idx || !out || !lse))
    return NSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256))
    return NSA_ERR_INVALID_ARG;
  Layout L;
  st = make_layout(dims, &L);
  if (st != NSA_OK) return st;
  if (workspace_bytes < L.fwd_end) return NSA_ERR_WORKSPACE;
  if (dims->total_tokens == 0) return NSA_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Params p;
  fill_params(&p, dims, L, workspace);
  p.q = q;
  p.k = k;
  p.v = v;
  p.sel = sel_idx;
  p.cu = cu_seqlens;
  p.out = out;
  p.lse = lse;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.window = window;
  st = run_index(dims, L, p, s);
  if (st != NSA_OK) return st;
  return cuda_status(launch_fwd(p, num_sms_cached(), L.max_wtiles, s, mark));
}

nsa_status nsa_sel_attn_fwd(const nsa_sel_attn_dims *dims, const void *q, const void *k,
                            const void *v, const int32_t *sel_idx, const int32_t *cu_seqlens,
                            float scale, void *out, float *lse, void *workspace,
                            size_t workspace_bytes, nsa_stream_t stream) {
  return fwd_impl(dims, q, k, v, sel_idx, cu_seqlens, scale, 0, out, lse, workspace,
                  workspace_bytes, stream);
}

nsa_status nsa_sel_attn_fwd_window(const nsa_sel_attn_dims *dims, const void *q, const void *k,
                                   const void *v, const int32_t *sel_idx,
                                   const int32_t *cu_seqlens, float scale, int window, void *out,
                                   float *lse, void *workspace, size_t workspace_bytes,
                                   nsa_stream_t stream) {
  if (window < 1) return NSA_ERR_INVALID_ARG;
  return fwd_impl(dims, q, k, v, sel_idx, cu_seqlens, scale, window, out, lse, workspace,
                  workspace_bytes, stream);
}

static nsa_status bwd_impl(const nsa_sel_attn_dims *dims, const void *q, const void *k,
                           const void *v, const int32_t *sel_idx, const int32_t *cu_seqlens,
                           float scale, int window, const void *out, const float *lse,
                           const void *dout, void *dq, void *dk, void *dv, void *workspace,
                           size_t workspace_bytes, int index_ready, nsa_stream_t stream) {
  nsa_status st = check_dims(dims, true);
  if (st != NSA_OK) return st;
  st = check_kernels(dims);
  if (st != NSA_OK) return st;
  if (!cu_seqlens || !workspace || !std::isfinite(scale)) return NSA_ERR_INVALID_ARG;
  if (dims->total_tokens > 0 &&
      (!q || !k || !v || !sel_idx || !out || !lse || !dout || !dq || !dk || !dv))
    return NSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256))
    return NSA_ERR_INVALID_ARG;
  Layout L;
  st = make_layout(dims, &L);
  if (st != NSA_OK) return st;
  if (workspace_bytes < L.bwd_end) return NSA_ERR_WORKSPACE;
  if (dims->total_tokens == 0) return NSA_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Params p;
  fill_params(&p, dims, L, workspace);
  p.q = q;
  p.k = k;
  p.v = v;
  p.sel = sel_idx;
  p.cu = cu_seqlens;
  p.out_in = out;
  p.lse_in = lse;
  p.dout = dout;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.window = window;
  if (!index_ready) {
    st = run_index(dims, L, p, s);
    if (st != NSA_OK) return st;
  }
  return cuda_status(launch_bwd(p, num_sms_cached(), L.max_wtiles, s, mark));
}

nsa_status nsa_sel_attn_bwd(const nsa_sel_attn_dims *dims, const void *q, const void *k,
                            const void *v, const int32_t *sel_idx, const int32_t *cu_seqlens,
                            float scale, const void *out, const float *lse, const void *dout,
                            void *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes,
                            int index_ready, nsa_stream_t stream) {
  return bwd_impl(dims, q, k, v, sel_idx, cu_seqlens, scale, 0, out, lse, dout, dq, dk, dv,
                  workspace, workspace_bytes, index_ready, stream);
}

nsa_status nsa_sel_attn_bwd_window(const nsa_sel_attn_dims *dims, const void *q, const void *k,
                                   const void *v, const int32_t *sel_idx,
                                   const int32_t *cu_seqlens, float scale, int window,
                                   const void *out, const float *lse, const void *dout, void *dq,
                                   void *dk, void *dv, void *workspace, size_t workspace_bytes,
                                   int index_ready, nsa_stream_t stream) {
  if (window < 1) return NSA_ERR_INVALID_ARG;
  return bwd_impl(dims, q, k, v, sel_idx, cu_seqlens, scale, window, out, lse, dout, dq, dk, dv,
                  workspace, workspace_bytes, index_ready, stream);
}

nsa_status nsa_sel_attn_window_select(const nsa_sel_attn_dims *dims, const int32_t *cu_seqlens,
                                      int window, int32_t *sel_idx, nsa_stream_t stream) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  if (!cu_seqlens || window < 1 || (dims->total_tokens > 0 && !sel_idx))
    return NSA_ERR_INVALID_ARG;
  // blocks that can hold keys of a window: ceil((window - 1) / B_K) + 1
  if (dims->topk < (window - 1 + dims->block_size - 1) / dims->block_size + 1)
    return NSA_ERR_INVALID_ARG;
  return cuda_status(launch_window_select(cu_seqlens, dims->num_seqs, dims->total_tokens,
                                          dims->h_k, dims->block_size, dims->topk, window,
                                          sel_idx, reinterpret_cast<cudaStream_t>(stream)));
}

nsa_status nsa_gate_combine_fwd(const nsa_sel_attn_dims *dims, int n_branch, const void *o0,
                                const void *o1, const void *o2, const float *gates, void *out,
                                nsa_stream_t stream) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  if (n_branch < 1 || n_branch > 3 || !gates || !out || !o0 || (n_branch > 1 && !o1) ||
      (n_branch > 2 && !o2))
    return NSA_ERR_INVALID_ARG;
  if (!aligned(o0, 4) || !aligned(o1, 4) || !aligned(o2, 4) || !aligned(out, 4) ||
      !aligned(gates, 4))
    return NSA_ERR_INVALID_ARG;
  return cuda_status(launch_gate_combine((int64_t)dims->total_tokens * dims->h_q, dims->head_dim,
                                         dims->dtype == NSA_FP16, n_branch, o0, o1, o2, gates,
                                         out, nullptr, nullptr, nullptr, nullptr, nullptr, false,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

nsa_status nsa_gate_combine_bwd(const nsa_sel_attn_dims *dims, int n_branch, const void *o0,
                                const void *o1, const void *o2, const float *gates,
                                const void *dout, void *do0, void *do1, void *do2,
                                float *dgates, nsa_stream_t stream) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  if (n_branch < 1 || n_branch > 3 || !gates || !dout || !dgates || !o0 ||
      (n_branch > 1 && !o1) || (n_branch > 2 && !o2))
    return NSA_ERR_INVALID_ARG;
  if (!aligned(o0, 4) || !aligned(o1, 4) || !aligned(o2, 4) || !aligned(dout, 4) ||
      !aligned(do0, 4) || !aligned(do1, 4) || !aligned(do2, 4) || !aligned(gates, 4) ||
      !aligned(dgates, 4))
    return NSA_ERR_INVALID_ARG;
  return cuda_status(launch_gate_combine((int64_t)dims->total_tokens * dims->h_q, dims->head_dim,
                                         dims->dtype == NSA_FP16, n_branch, o0, o1, o2, gates,
                                         nullptr, dout, do0, do1, do2, dgates, true,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

nsa_status nsa_sel_attn_staging_size(const nsa_sel_attn_dims *dims, size_t *bytes) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  if (!bytes) return NSA_ERR_INVALID_ARG;
  const size_t N = dims->total_tokens, d = dims->head_dim;
  const size_t qb = align256(N * dims->h_q * d * 2), kb = align256(N * dims->h_k * d * 2);
  const size_t selb = align256(4 * N * dims->h_k * dims->topk);
  const size_t cub = align256(4 * static_cast<size_t>(dims->num_seqs + 1));
  const size_t lseb = align256(4 * N * dims->h_q);
  // q, k, v, dout, sel, cu, out, lse, dq, dk, dv
  *bytes = 3 * qb + 4 * kb + selb + cub + lseb + qb;
  return NSA_OK;
}

// Side stream and events of nsa_sel_attn_step_host, one set per device, created on
// first use and kept for the life of the process.
struct StepAux {
  int device = -1;
  cudaStream_t side = nullptr;
  cudaEvent_t dout_in = nullptr, fwd_done = nullptr, out_back = nullptr;
  cudaEvent_t kv_in = nullptr, q_in = nullptr;
};
static bool step_aux(StepAux **aux) {
  static std::mutex mu;
  static std::vector<StepAux> all;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (auto &a : all)
    if (a.device == dev) {
      *aux = &a;
      return true;
    }
  StepAux a;
  a.device = dev;
  if (cudaStreamCreateWithFlags(&a.side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&a.dout_in, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&a.fwd_done, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&a.out_back, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&a.kv_in, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&a.q_in, cudaEventDisableTiming) != cudaSuccess)
    return false;
  all.reserve(16);
  all.push_back(a);
  *aux = &all.back();
  return true;
}

nsa_status nsa_sel_attn_step_host(const nsa_sel_attn_dims *dims, const void *host_q,
                                  const void *host_k, const void *host_v,
                                  const int32_t *host_sel_idx, const int32_t *host_cu_seqlens,
                                  const void *host_dout, float scale, void *host_out,
                                  float *host_lse, void *host_dq, void *host_dk, void *host_dv,
                                  void *staging, size_t staging_bytes, void *workspace,
                                  size_t workspace_bytes, nsa_stream_t stream) {
  nsa_status st = check_dims(dims, true);
  if (st != NSA_OK) return st;
  size_t need = 0;
  nsa_sel_attn_staging_size(dims, &need);
  if (!staging || staging_bytes < need || !aligned(staging, 256)) return NSA_ERR_INVALID_ARG;
  if (!host_cu_seqlens) return NSA_ERR_INVALID_ARG;
  const size_t N = dims->total_tokens, d = dims->head_dim;
  if (N > 0 && (!host_q || !host_k || !host_v || !host_sel_idx || !host_dout || !host_out ||
                !host_dq || !host_dk || !host_dv))
    return NSA_ERR_INVALID_ARG;
  const size_t qbytes = N * dims->h_q * d * 2, kbytes = N * dims->h_k * d * 2;
  const size_t selbytes = 4 * N * dims->h_k * dims->topk;
  const size_t cubytes = 4 * static_cast<size_t>(dims->num_seqs + 1), lsebytes = 4 * N * dims->h_q;
  char *w = static_cast<char *>(staging);
  size_t o = 0;
  auto take = [&](size_t b) {
    char *at = w + o;
    o += align256(b);
    return at;
  };
  char *q = take(qbytes), *k = take(kbytes), *v = take(kbytes), *dout = take(qbytes);
  char *sel = take(selbytes), *cu = take(cubytes), *out = take(qbytes);
  char *lse = take(lsebytes), *dq = take(qbytes), *dk = take(kbytes), *dv = take(kbytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  StepAux *aux = nullptr;
  if (!step_aux(&aux)) return NSA_ERR_CUDA;
  cudaStream_t s2 = aux->side;
  // The forward's inputs go first, split over the two streams: k and v on the side
  // stream, sel, cu_seqlens and q on the caller's.  dout follows on the side stream
  // once q has landed, so that it shares the host link with the forward's compute
  // rather than with the forward's inputs.  out and lse travel back on the side stream
  // while the backward runs; the gradients go back split over the two streams.
  struct Copy { void *dst; const void *src; size_t n; };
  auto copies = [](const Copy *c, int nc, cudaMemcpyKind kind, cudaStream_t st_) {
    for (int i = 0; i < nc; ++i)
      if (c[i].n && cudaMemcpyAsync(c[i].dst, c[i].src, c[i].n, kind, st_) != cudaSuccess)
        return false;
    return true;
  };
  auto join = [](cudaEvent_t ev, cudaStream_t from, cudaStream_t to) {   // to waits for from
    return cudaEventRecord(ev, from) == cudaSuccess &&
           cudaStreamWaitEvent(to, ev, 0) == cudaSuccess;
  };
  const Copy in_kv[] = {{k, host_k, kbytes}, {v, host_v, kbytes}};
  const Copy in_q[] = {{sel, host_sel_idx, selbytes}, {cu, host_cu_seqlens, cubytes},
                       {q, host_q, qbytes}};
  const Copy in_do[] = {{dout, host_dout, qbytes}};
  if (!join(aux->fwd_done, s, s2) ||                       // s2 after s's earlier work
      !copies(in_kv, 2, cudaMemcpyHostToDevice, s2) ||
      cudaEventRecord(aux->kv_in, s2) != cudaSuccess ||
      !copies(in_q, 3, cudaMemcpyHostToDevice, s) || !join(aux->q_in, s, s2) ||
      !copies(in_do, 1, cudaMemcpyHostToDevice, s2) ||
      cudaEventRecord(aux->dout_in, s2) != cudaSuccess ||
      cudaStreamWaitEvent(s, aux->kv_in, 0) != cudaSuccess)
    return NSA_ERR_CUDA;
  st = nsa_sel_attn_fwd(dims, q, k, v, reinterpret_cast<int32_t *>(sel),
                        reinterpret_cast<int32_t *>(cu), scale, out, reinterpret_cast<float *>(lse),
                        workspace, workspace_bytes, stream);
  if (st != NSA_OK) return st;
  const Copy back1[] = {{host_out, out, qbytes}, {host_lse, lse, host_lse ? lsebytes : 0}};
  if (!join(aux->fwd_done, s, s2) || !copies(back1, 2, cudaMemcpyDeviceToHost, s2) ||
      cudaEventRecord(aux->out_back, s2) != cudaSuccess ||
      cudaStreamWaitEvent(s, aux->dout_in, 0) != cudaSuccess)
    return NSA_ERR_CUDA;
  t_dkv_ready = aux->kv_in;
  t_dkv_recorded = false;
  st = nsa_sel_attn_bwd(dims, q, k, v, reinterpret_cast<int32_t *>(sel),
                        reinterpret_cast<int32_t *>(cu), scale, out, reinterpret_cast<float *>(lse),
                        dout, dq, dk, dv, workspace, workspace_bytes, 1, stream);
  t_dkv_ready = nullptr;
  if (st != NSA_OK) return st;
  // dk and dv go down on the side stream once their reduction is done, while the dQ
  // reduction still runs; without that record, after the whole backward
  if (!t_dkv_recorded && cudaEventRecord(aux->kv_in, s) != cudaSuccess) return NSA_ERR_CUDA;
  const Copy back_kv[] = {{host_dk, dk, kbytes}, {host_dv, dv, kbytes}};
  const Copy back_q[] = {{host_dq, dq, qbytes}};
  if (cudaStreamWaitEvent(s2, aux->kv_in, 0) != cudaSuccess ||
      !copies(back_kv, 2, cudaMemcpyDeviceToHost, s2) ||
      cudaEventRecord(aux->kv_in, s2) != cudaSuccess ||
      !copies(back_q, 1, cudaMemcpyDeviceToHost, s) ||
      cudaStreamWaitEvent(s, aux->kv_in, 0) != cudaSuccess)   // after out, lse, dk and dv
    return NSA_ERR_CUDA;
  return cuda_status(cudaStreamSynchronize(s));
}

nsa_status nsa_sel_attn_decode(const nsa_sel_attn_dims *dims, const void *q, const void *k_cache,
                               const void *v_cache, const int32_t *sel_idx,
                               const int32_t *cu_seqlens, float scale, void *out, float *lse,
                               int32_t *device_status, nsa_stream_t stream) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  if (!(dims->head_dim == 64 || dims->head_dim == 128)) return NSA_ERR_UNSUPPORTED;
  if (dims->h_q / dims->h_k > 16) return NSA_ERR_UNSUPPORTED;
  if ((int64_t)dims->num_seqs * dims->h_q >= (int64_t(1) << 31)) return NSA_ERR_UNSUPPORTED;
  if (!cu_seqlens || !q || !sel_idx || !out || !lse) return NSA_ERR_INVALID_ARG;
  if (dims->total_tokens > 0 && (!k_cache || !v_cache)) return NSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || (device_status && !aligned(device_status, 4)))
    return NSA_ERR_INVALID_ARG;
  return cuda_status(launch_decode(dims->num_seqs, dims->h_q, dims->h_k, dims->head_dim,
                                   dims->block_size, dims->topk, dims->dtype == NSA_FP16, scale,
                                   q, k_cache, v_cache, sel_idx, cu_seqlens, out, lse,
                                   device_status, reinterpret_cast<cudaStream_t>(stream)));
}

static nsa_status check_cmp(const nsa_sel_attn_dims *dims, int kernel_size, int kernel_stride) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  if (!(dims->head_dim == 64 || dims->head_dim == 128)) return NSA_ERR_UNSUPPORTED;
  if (kernel_stride < 1 || kernel_size < kernel_stride) return NSA_ERR_INVALID_ARG;
  if (dims->h_q / dims->h_k > 128) return NSA_ERR_UNSUPPORTED;
  return NSA_OK;
}

nsa_status nsa_compress_kv(const nsa_sel_attn_dims *dims, const int32_t *cu_seqlens,
                           int kernel_size, int kernel_stride, const void *k, const void *v,
                           void *kc, void *vc, int32_t *cu_cmp, int32_t *device_status,
                           nsa_stream_t stream) {
  nsa_status st = check_cmp(dims, kernel_size, kernel_stride);
  if (st != NSA_OK) return st;
  const int64_t rows_cap = dims->total_tokens / kernel_stride;
  if (!cu_seqlens || !cu_cmp) return NSA_ERR_INVALID_ARG;
  if (rows_cap > 0 && (!k || !v || !kc || !vc)) return NSA_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(kc, 16) || !aligned(vc, 16) ||
      !aligned(cu_cmp, 4) || (device_status && !aligned(device_status, 4)))
    return NSA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_cmp_offsets(cu_seqlens, dims->num_seqs, dims->total_tokens, kernel_size,
                                     kernel_stride, cu_cmp, device_status, s);
  if (e != cudaSuccess) return NSA_ERR_CUDA;
  return cuda_status(launch_compress(dims->head_dim, dims->dtype == NSA_FP16, cu_seqlens, cu_cmp,
                                     dims->num_seqs, dims->total_tokens, dims->h_k, kernel_size,
                                     kernel_stride, rows_cap, k, v, kc, vc, s));
}

// Launch shape of nsa_cmp_attn_select: tokens per CTA and the workspace bytes that
// the importance rows take in global memory (0 when shared memory holds them in a
// CTA of full size, or when no workspace is offered).
static nsa_status cmp_plan(const nsa_sel_attn_dims *dims, int max_seqlen, bool ws_ok, int *tt,
                           int *nb_max, size_t *ws_bytes) {
  const int g = dims->h_q / dims->h_k;
  const int64_t nb = ((int64_t)max_seqlen + dims->block_size - 1) / dims->block_size;
  if (nb > (int64_t(1) << 20)) return NSA_ERR_UNSUPPORTED;
  *nb_max = static_cast<int>(nb);
  const int tt_smem = cmp_tokens_per_cta(dims->head_dim, g, *nb_max, true);
  const int tt_full = cmp_tokens_per_cta(dims->head_dim, g, *nb_max, false);
  *ws_bytes = 0;
  if (tt_smem == tt_full || !ws_ok) {
    *tt = tt_smem;
    return tt_smem ? NSA_OK : NSA_ERR_UNSUPPORTED;
  }
  *tt = tt_full;
  const int64_t ctas = ((int64_t)dims->total_tokens + tt_full - 1) / tt_full * dims->h_k;
  *ws_bytes = static_cast<size_t>(ctas) * tt_full * (*nb_max) * sizeof(float);
  return NSA_OK;
}

nsa_status nsa_cmp_workspace_size(const nsa_sel_attn_dims *dims, int kernel_size,
                                  int kernel_stride, int max_seqlen, size_t *bytes) {
  nsa_status st = check_cmp(dims, kernel_size, kernel_stride);
  if (st != NSA_OK) return st;
  if (max_seqlen < 1 || !bytes) return NSA_ERR_INVALID_ARG;
  int tt = 0, nb = 0;
  return cmp_plan(dims, max_seqlen, true, &tt, &nb, bytes);
}

nsa_status nsa_cmp_attn_select(const nsa_sel_attn_dims *dims, const void *q, const void *kc,
                               const void *vc, const int32_t *cu_seqlens, const int32_t *cu_cmp,
                               int kernel_size, int kernel_stride, int max_seqlen, float scale,
                               int init_blocks, int local_blocks, void *out, float *lse,
                               int32_t *sel_idx, int32_t *device_status, void *workspace,
                               size_t workspace_bytes, nsa_stream_t stream) {
  nsa_status st = check_cmp(dims, kernel_size, kernel_stride);
  if (st != NSA_OK) return st;
  if (max_seqlen < 1 || init_blocks < 0 || local_blocks < 0 || !(scale > 0.f))
    return NSA_ERR_INVALID_ARG;
  if (!cu_seqlens || !cu_cmp) return NSA_ERR_INVALID_ARG;
  if (dims->total_tokens > 0 && (!q || !out || !lse || !sel_idx)) return NSA_ERR_INVALID_ARG;
  const int64_t rows_cap = dims->total_tokens / kernel_stride;
  if (rows_cap > 0 && (!kc || !vc)) return NSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kc, 16) || !aligned(vc, 16) || !aligned(out, 16) ||
      !aligned(lse, 4) || !aligned(sel_idx, 4) || (device_status && !aligned(device_status, 4)))
    return NSA_ERR_INVALID_ARG;
  const int g = dims->h_q / dims->h_k;
  if (workspace && !aligned(workspace, 16)) return NSA_ERR_INVALID_ARG;
  int tt = 0, nb_max = 0;
  size_t ws_need = 0;
  st = cmp_plan(dims, max_seqlen, workspace != nullptr, &tt, &nb_max, &ws_need);
  if (st != NSA_OK) return st;
  if (ws_need > workspace_bytes) return NSA_ERR_WORKSPACE;
  CmpParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.kc = kc;
  p.vc = vc;
  p.cu = cu_seqlens;
  p.cu_cmp = cu_cmp;
  p.num_seqs = dims->num_seqs;
  p.n = dims->total_tokens;
  p.h_q = dims->h_q;
  p.h_k = dims->h_k;
  p.g = g;
  p.ksize = kernel_size;
  p.stride = kernel_stride;
  p.block = dims->block_size;
  p.topk = dims->topk;
  p.init_blocks = init_blocks;
  p.local_blocks = local_blocks;
  p.max_seqlen = max_seqlen;
  p.tt = tt;
  p.nb_max = nb_max;
  p.rows_cap = rows_cap;
  p.imp_ws = ws_need ? static_cast<float *>(workspace) : nullptr;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = out;
  p.lse = lse;
  p.sel = sel_idx;
  p.status = device_status;
  return cuda_status(launch_cmp_select(dims->head_dim, dims->dtype == NSA_FP16, p,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

nsa_status nsa_sel_attn_get_status(const nsa_sel_attn_dims *dims, void *workspace,
                                   nsa_stream_t stream, int32_t *bits) {
  nsa_status st = check_dims(dims, false);
  if (st != NSA_OK) return st;
  if (!workspace) return NSA_ERR_INVALID_ARG;
  Layout L;
  st = make_layout(dims, &L);
  if (st != NSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t word = 0;
  char *w = static_cast<char *>(workspace);
  if (cudaMemcpyAsync(&word, w + L.status, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return NSA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return NSA_ERR_CUDA;
  if (cudaMemsetAsync(w + L.status, 0, 4, s) != cudaSuccess) return NSA_ERR_CUDA;
  if (bits) *bits = word;
  if (word & NSA_DEVERR_TIMEOUT) return NSA_ERR_TIMEOUT;
  if (word & (NSA_DEVERR_BAD_INDEX | NSA_DEVERR_BAD_SEQLENS)) return NSA_ERR_BAD_INDEX;
  return NSA_OK;
}

int32_t nsa_sel_attn_num_kernels(void) { return kNumKernels; }

const char *nsa_sel_attn_kernel_name(int32_t id) {
  return (id >= 0 && id < kNumKernels) ? kKernelNames[id] : "unknown";
}

nsa_status nsa_sel_attn_profile_enable(int32_t on) {
  g_prof.on = on != 0;
  return NSA_OK;
}

nsa_status nsa_sel_attn_profile_collect(int32_t *launches, float *total_ms) {
  if (!launches || !total_ms) return NSA_ERR_INVALID_ARG;
  for (int i = 0; i < kNumKernels; ++i) {
    launches[i] = 0;
    total_ms[i] = 0.f;
  }
  nsa_status st = NSA_OK;
  for (const Rec &r : g_prof.recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) {
      st = NSA_ERR_CUDA;
      continue;
    }
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      st = NSA_ERR_CUDA;
      continue;
    }
    launches[r.id] += 1;
    total_ms[r.id] += ms;
  }
  g_prof.recs.clear();
  g_prof.used = 0;
  g_prof.pending = nullptr;
  return st;
}

const char *nsa_status_string(nsa_status status) {
  switch (status) {
    case NSA_OK: return "ok";
    case NSA_ERR_INVALID_ARG: return "invalid argument";
    case NSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case NSA_ERR_WORKSPACE: return "workspace too small";
    case NSA_ERR_CUDA: return "CUDA error";
    case NSA_ERR_BAD_INDEX: return "invalid selection index or sequence offsets seen on device";
    case NSA_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
