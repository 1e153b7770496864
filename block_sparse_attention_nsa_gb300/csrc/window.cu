// window.cu -- the sliding-window branch's selection and the gated combination of
// the branches (Native Sparse Attention's three parallel branches: compressed,
// selected and sliding-window attention, per the papernotes page's 领域现状 and the
// Flash-Sparse-Attention README's "Usage", window_size = 512).
//
// The sliding window runs on the selected-attention kernels: a token's window of
// keys (tau - window, tau] is a set of consecutive blocks, written here as a
// selection row, and the attention kernels add the window's lower key bound to the
// causal mask (Params::window).  The combination out = sum_b gate_b * o_b is an
// elementwise pass over the branch outputs (HBM-bound; one warp per row).
#include "common.cuh"

namespace nsa {

// One thread per token: the blocks holding keys (tau - window, tau], newest first,
// the other slots -1, for every KV head.
__global__ void __launch_bounds__(256) window_select_kernel(const int32_t *cu, int num_seqs,
                                                            int n, int h_k, int block,
                                                            int topk, int window,
                                                            int32_t *sel) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n) return;
  const int s = seq_of(cu, num_seqs, t);
  const int tau = t - cu[s];
  const int c = tau / block;
  const int first = tau - window + 1 > 0 ? (tau - window + 1) / block : 0;
  for (int h = 0; h < h_k; ++h) {
    int32_t *row = sel + ((int64_t)h * n + t) * topk;
    for (int k = 0; k < topk; ++k) row[k] = (c - k >= first) ? c - k : -1;
  }
}

// out[r] = sum_b gates[r][b] o_b[r], one warp per row r = (token, query head).
template <int D, bool kFp16>
__global__ void __launch_bounds__(256) gate_combine_kernel(int64_t rows, int nbr,
                                                           const void *o0, const void *o1,
                                                           const void *o2, const float *gates,
                                                           void *out) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint16_t *src[3] = {static_cast<const uint16_t *>(o0), static_cast<const uint16_t *>(o1),
                            static_cast<const uint16_t *>(o2)};
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int b = 0; b < nbr; ++b) {
    const float gt = gates[r * nbr + b];
    const uint16_t *x = src[b] + r * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 f = unpack2<kFp16>(*reinterpret_cast<const uint32_t *>(x + e));
      acc[e] = fmaf(gt, f.x, acc[e]);
      acc[e + 1] = fmaf(gt, f.y, acc[e + 1]);
    }
  }
  uint16_t *y = static_cast<uint16_t *>(out) + r * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    *reinterpret_cast<uint32_t *>(y + e) = pack2<kFp16>(acc[e], acc[e + 1]);
}

// d o_b[r] = gates[r][b] dout[r]; d gates[r][b] = sum_d dout[r] o_b[r] (fp32 sums).
template <int D, bool kFp16>
__global__ void __launch_bounds__(256) gate_combine_bwd_kernel(
    int64_t rows, int nbr, const void *o0, const void *o1, const void *o2, const float *gates,
    const void *dout, void *d0, void *d1, void *d2, float *dgates) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint16_t *src[3] = {static_cast<const uint16_t *>(o0), static_cast<const uint16_t *>(o1),
                            static_cast<const uint16_t *>(o2)};
  uint16_t *dst[3] = {static_cast<uint16_t *>(d0), static_cast<uint16_t *>(d1),
                      static_cast<uint16_t *>(d2)};
  float dy[E];
  const uint16_t *gy = static_cast<const uint16_t *>(dout) + r * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const float2 f = unpack2<kFp16>(*reinterpret_cast<const uint32_t *>(gy + e));
    dy[e] = f.x;
    dy[e + 1] = f.y;
  }
  for (int b = 0; b < nbr; ++b) {
    const float gt = gates[r * nbr + b];
    const uint16_t *x = src[b] + r * D + lane * E;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < E; e += 2) {
      const float2 f = unpack2<kFp16>(*reinterpret_cast<const uint32_t *>(x + e));
      dot = fmaf(dy[e], f.x, fmaf(dy[e + 1], f.y, dot));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    if (lane == 0) dgates[r * nbr + b] = dot;
    if (dst[b]) {
      uint16_t *y = dst[b] + r * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; e += 2)
        *reinterpret_cast<uint32_t *>(y + e) = pack2<kFp16>(gt * dy[e], gt * dy[e + 1]);
    }
  }
}

cudaError_t launch_window_select(const int32_t *cu, int num_seqs, int n, int h_k, int block,
                                 int topk, int window, int32_t *sel, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  window_select_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
      cu, num_seqs, n, h_k, block, topk, window, sel);
  return cudaGetLastError();
}

template <int D, bool kFp16>
static cudaError_t run_combine(int64_t rows, int nbr, const void *o0, const void *o1,
                               const void *o2, const float *gates, void *out, const void *dout,
                               void *d0, void *d1, void *d2, float *dgates, bool bwd,
                               cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((rows + 7) / 8);
  if (bwd)
    gate_combine_bwd_kernel<D, kFp16><<<grid, 256, 0, s>>>(rows, nbr, o0, o1, o2, gates, dout, d0,
                                                           d1, d2, dgates);
  else
    gate_combine_kernel<D, kFp16><<<grid, 256, 0, s>>>(rows, nbr, o0, o1, o2, gates, out);
  return cudaGetLastError();
}

cudaError_t launch_gate_combine(int64_t rows, int d, bool fp16, int nbr, const void *o0,
                                const void *o1, const void *o2, const float *gates, void *out,
                                const void *dout, void *d0, void *d1, void *d2, float *dgates,
                                bool bwd, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  switch (d) {
    case 64:
      return fp16 ? run_combine<64, true>(rows, nbr, o0, o1, o2, gates, out, dout, d0, d1, d2,
                                          dgates, bwd, s)
                  : run_combine<64, false>(rows, nbr, o0, o1, o2, gates, out, dout, d0, d1, d2,
                                           dgates, bwd, s);
    case 128:
      return fp16 ? run_combine<128, true>(rows, nbr, o0, o1, o2, gates, out, dout, d0, d1, d2,
                                           dgates, bwd, s)
                  : run_combine<128, false>(rows, nbr, o0, o1, o2, gates, out, dout, d0, d1, d2,
                                            dgates, bwd, s);
    case 256:
      return fp16 ? run_combine<256, true>(rows, nbr, o0, o1, o2, gates, out, dout, d0, d1, d2,
                                           dgates, bwd, s)
                  : run_combine<256, false>(rows, nbr, o0, o1, o2, gates, out, dout, d0, d1, d2,
                                            dgates, bwd, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nsa
