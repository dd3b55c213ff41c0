// Exact prefetch cap, shared by the indexer's fix-up kernel and the top-k kernel.
//
// "ECHO: Efficient KV Cache Offloading with Lossless Prefetching ..." review page,
// "Decode: predict the transfer, then recall exactly": a counter caps the prefetch
// volume.  The cap is applied to the first cap qualifying tokens by ascending token
// index (so the prefetched set is deterministic).  The indexer claims staging rows
// optimistically, in any order; for the rare request whose qualifying tokens
// outnumber its cap, pf_fixup_block re-derives the first-cap set from the stored
// scores and swaps wrongly staged tokens for missing ones, reusing their rows.
#pragma once

#include "common.cuh"

namespace echo {

// What the fix-up of one request reads and writes (all device pointers).
struct PfFix {
  const int32_t *seq_len;
  int Lmax;
  const int32_t *cap;       // null: no prefetch, nothing to fix
  int cap_max;
  const int32_t *host_base;
  echo_cache_layer_t L;
  const float *scores;      // [B, Lmax] indexer scores of this step
  int32_t *pf_list;         // [B * cap_max], indexed by staging row
  int32_t *pf_count;        // [B]: qualifying count in, min(qualifying, cap) out
  void *stage_kv;           // [B * cap_max, 576] staging rows
};

constexpr int FX_THREADS = 512;      // pf_fixup_block needs exactly this many threads
constexpr int FX_LIST = 2048;

struct PfFixSmem {
  int32_t need_t[FX_LIST], free_row[FX_LIST], free_t[FX_LIST];
  int32_t seg_pre[FX_THREADS + 1];
  int n_need, n_free;
};

static __device__ __forceinline__ bool pf_fixup_needed(const PfFix &P, int b) {
  return P.cap != nullptr && P.pf_count[b] > min(P.cap[b], P.cap_max);
}

// One request's exact-cap fix-up, run by a whole block of FX_THREADS threads with
// sm as shared scratch.  theta is the threshold the indexer scored against.
// Qualifying = score > theta and not resident at scoring time (host2gpu < 0).
// On return pf_count[b] = min(qualifying, cap).  Every thread of the block must
// call it (it synchronises the block); it returns at once when there is nothing to fix.
static __device__ __noinline__ void pf_fixup_block(const PfFix &P, int b, float theta, PfFixSmem &sm) {
  if (!pf_fixup_needed(P, b)) return;
  const int cap = min(P.cap[b], P.cap_max);
  const echo_cache_layer_t &L = P.L;
  const int Lb = min(P.seq_len[b], P.Lmax);
  const int64_t base = P.host_base[b];
  const float *sc = P.scores + (int64_t)b * P.Lmax;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr int NW = FX_THREADS / 32;
  // warp w owns the 32-aligned token segment [w0, w1); its lanes read consecutive
  // tokens (coalesced), four chunks of 32 per iteration with their loads issued
  // together, and the qualifiers' ranks follow from per-warp counts
  const int wseg = ((Lb + NW - 1) / NW + 31) & ~31;
  const int w0 = min(Lb, warp * wseg), w1 = min(Lb, w0 + wseg);
  const int esz = L.kv_dtype == ECHO_F32 ? 4 : 2;
  // qualifier test of token t with its map entry g (resident at scoring time: not one)
  auto load4 = [&](int t0, bool (&q)[4], int32_t (&g)[4]) {
    float v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = t0 + 32 * j + lane;
      v[j] = t < w1 ? sc[t] : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = t0 + 32 * j + lane;
      const bool above = t < w1 && v[j] > theta;
      g[j] = above ? L.host2gpu[base + t] : 0;
      q[j] = above && g[j] < 0;
    }
  };
  for (int round = 0; round < 64; ++round) {
    uint32_t c = 0;
    for (int t0 = w0; t0 < w1; t0 += 128) {
      bool q[4];
      int32_t g[4];
      load4(t0, q, g);
#pragma unroll
      for (int j = 0; j < 4; ++j) c += __popc(__ballot_sync(0xffffffffu, q[j]));
    }
    if (lane == 0) sm.seg_pre[warp] = (int32_t)c;
    if (tid == 0) { sm.n_need = 0; sm.n_free = 0; }
    __syncthreads();
    uint32_t r = 0;
    for (int w = 0; w < warp; ++w) r += (uint32_t)sm.seg_pre[w];
    for (int t0 = w0; t0 < w1; t0 += 128) {
      bool q[4];
      int32_t g[4];
      load4(t0, q, g);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t bal = __ballot_sync(0xffffffffu, q[j]);
        const uint32_t rk = r + __popc(bal & lanemask_lt());
        const int t = t0 + 32 * j + lane;
        if (q[j] && rk < (uint32_t)cap && g[j] == -1) {
          const int i = atomicAdd(&sm.n_need, 1);
          if (i < FX_LIST) sm.need_t[i] = t;
        } else if (q[j] && rk >= (uint32_t)cap && g[j] <= -2) {
          const int i = atomicAdd(&sm.n_free, 1);
          if (i < FX_LIST) { sm.free_row[i] = -2 - g[j]; sm.free_t[i] = t; }
        }
        r += __popc(bal);
      }
    }
    __syncthreads();
    const int np = min(min(sm.n_need, sm.n_free), FX_LIST);
    if (np == 0) break;
    // swap: the dropped token returns to "host only", the added one takes its row
    for (int i = tid; i < np; i += FX_THREADS) {
      const int row = sm.free_row[i];
      L.host2gpu[base + sm.free_t[i]] = -1;
      L.host2gpu[base + sm.need_t[i]] = -2 - row;
      P.pf_list[row] = sm.need_t[i];
    }
    __syncthreads();
    for (int i0 = warp * 4; i0 < np; i0 += NW * 4) {
      const uint4 *src[4] = {nullptr, nullptr, nullptr, nullptr};
      uint4 *dst[4] = {nullptr, nullptr, nullptr, nullptr};
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + j;
        if (i >= np) break;
        src[j] = reinterpret_cast<const uint4 *>((const char *)L.host_kv + (base + sm.need_t[i]) * KV_W * esz);
        dst[j] = reinterpret_cast<uint4 *>((char *)P.stage_kv + (int64_t)sm.free_row[i] * KV_W * esz);
      }
      warp_copy_rows4(src, dst, KV_W * esz / 16);
    }
    // every wrongly staged token gave its row to a missing one, and the lists held them
    // all: the staged set is the first-cap set, no rescan needed
    const bool done = sm.n_need == sm.n_free && sm.n_need <= FX_LIST;
    __syncthreads();
    if (done) break;
  }
  if (tid == 0) P.pf_count[b] = cap;
}

}  // namespace echo
