// Block-sparse selection (N4): the block scores that the exact top-k selects blocks
// from, and the token slots of the selected blocks for sparse MLA.
//
// "ECHO: Efficient KV Cache Offloading with Lossless Prefetching ..." review page,
// critique section: the design adapts to block-sparse / GQA models by keeping the
// cache metadata per block of tokens.  A block of T consecutive tokens is one host
// index and one GPU slot (the layer's block_tokens); its score is the largest of its
// tokens' indexer scores.

#include <algorithm>

#include "common.cuh"

namespace echo {

// Blocks of T >= 32 tokens: one warp per (request, block), the largest score of the
// block's tokens below the request's length.  The first warp of each row writes the
// request's block count.
__global__ void block_scores_warp_kernel(const float *scores, const int32_t *seq_len, int B, int Lmax, int T,
                                         int nbmax, float *bscores, int32_t *seq_len_blk) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  if (w >= (int64_t)B * nbmax) return;
  const int b = (int)(w / nbmax), j = (int)(w % nbmax);
  const int L = min(max(seq_len[b], 0), Lmax);
  const int nb = (L + T - 1) / T;
  if (j == 0 && lane == 0) seq_len_blk[b] = nb;
  if (j >= nb) return;
  const float *row = scores + (int64_t)b * Lmax;
  float m = -INFINITY;
  for (int t = j * T + lane; t < min(L, j * T + T); t += 32) m = fmaxf(m, row[t]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) bscores[(int64_t)b * nbmax + j] = m;
}

// Blocks of T < 32 tokens: one thread per (request, block), grid-strided.
__global__ void block_scores_thread_kernel(const float *scores, const int32_t *seq_len, int B, int Lmax, int T,
                                           int nbmax, float *bscores, int32_t *seq_len_blk) {
  const int64_t n = (int64_t)B * nbmax;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(i / nbmax), j = (int)(i % nbmax);
    const int L = min(max(seq_len[b], 0), Lmax);
    const int nb = (L + T - 1) / T;
    if (j == 0) seq_len_blk[b] = nb;
    if (j >= nb) continue;
    const float *row = scores + (int64_t)b * Lmax;
    float m = -INFINITY;
    for (int t = j * T; t < min(L, j * T + T); ++t) m = fmaxf(m, row[t]);
    bscores[i] = m;
  }
}

// One thread per token position of the selected blocks.
__global__ void expand_slots_kernel(const int32_t *sel_blk, const int32_t *block_slot, const int32_t *seq_len, int B,
                                    int kb, int T, int32_t *out) {
  const int64_t n = (int64_t)B * kb * T;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i / T;                   // (request, selected block) entry
    const int b = (int)(e / kb), t = (int)(i % T);
    const int32_t j = sel_blk[e], g = block_slot[e];
    out[i] = (j >= 0 && g >= 0 && (int64_t)j * T + t < seq_len[b]) ? g * T + t : -1;
  }
}

}  // namespace echo

using namespace echo;

extern "C" echo_status_t echo_block_scores(const float *scores, const int32_t *seq_len, int32_t B, int32_t Lmax,
                                           int32_t T, float *bscores, int32_t *seq_len_blk, echo_stream_t stream) {
  if (!scores || !seq_len || !bscores || !seq_len_blk || B <= 0 || Lmax <= 0 || T <= 0) return ECHO_ERR_INVALID_ARG;
  const int nbmax = (Lmax + T - 1) / T;
  cudaStream_t st = (cudaStream_t)stream;
  if (T >= 32) {
    const int64_t threads = (int64_t)B * nbmax * 32;
    block_scores_warp_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(scores, seq_len, B, Lmax, T, nbmax,
                                                                                bscores, seq_len_blk);
  } else {
    const int64_t n = (int64_t)B * nbmax;
    const int grid = (int)std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 8);
    block_scores_thread_kernel<<<grid, 256, 0, st>>>(scores, seq_len, B, Lmax, T, nbmax, bscores, seq_len_blk);
  }
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

extern "C" echo_status_t echo_expand_block_slots(const int32_t *sel_blk, const int32_t *block_slot,
                                                 const int32_t *seq_len, int32_t B, int32_t kb, int32_t T,
                                                 int32_t *out, echo_stream_t stream) {
  if (!sel_blk || !block_slot || !seq_len || !out || B <= 0 || kb <= 0 || T <= 0) return ECHO_ERR_INVALID_ARG;
  const int64_t n = (int64_t)B * kb * T;
  const int grid = (int)std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 8);
  expand_slots_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(sel_blk, block_slot, seq_len, B, kb, T, out);
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}
