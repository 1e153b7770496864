// compress.cuh -- launch parameters of the compressed branch and block selection
// (compress.cu), shared with the C ABI.
#pragma once
#include "common.cuh"

namespace nsa {

struct CmpParams {
  const void *q, *kc, *vc;
  const int32_t *cu, *cu_cmp;
  int num_seqs, n, h_q, h_k, g;
  int ksize, stride, block, topk, init_blocks, local_blocks;
  int max_seqlen, tt, nb_max;
  int64_t rows_cap;   // rows allocated for kc / vc
  float *imp_ws;      // importance rows in global memory (tt * nb_max per CTA), or null
  float scale_log2;
  void *out;
  float *lse;
  int32_t *sel;
  int32_t *status;
};

}  // namespace nsa
