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
  const int tid = threadIdx.x, warp = tid >> 5;
  constexpr int NW = FX_THREADS / 32;
  // thread tid owns the contiguous token segment [t0, t1): independent loads, and
  // its qualifiers' ranks follow from a block scan of the per-thread counts
  const int seg = (Lb + FX_THREADS - 1) / FX_THREADS;
  const int t0 = min(Lb, tid * seg), t1 = min(Lb, t0 + seg);
  const int esz = L.kv_dtype == ECHO_F32 ? 4 : 2;
  for (int round = 0; round < 64; ++round) {
    int c = 0;
#pragma unroll 8
    for (int t = t0; t < t1; ++t)
      if (sc[t] > theta && L.host2gpu[base + t] < 0) ++c;
    block_prefix(FX_THREADS, [&](int) { return c; }, sm.seg_pre);   // f(i) is evaluated by thread i
    if (tid == 0) { sm.n_need = 0; sm.n_free = 0; }
    __syncthreads();
    uint32_t r = sm.seg_pre[tid];
    for (int t = t0; t < t1; ++t) {
      if (!(sc[t] > theta)) continue;
      const int32_t g = L.host2gpu[base + t];
      if (g >= 0) continue;                            // resident at scoring time: not a qualifier
      if (r < (uint32_t)cap && g == -1) {
        const int i = atomicAdd(&sm.n_need, 1);
        if (i < FX_LIST) sm.need_t[i] = t;
      } else if (r >= (uint32_t)cap && g <= -2) {
        const int i = atomicAdd(&sm.n_free, 1);
        if (i < FX_LIST) { sm.free_row[i] = -2 - g; sm.free_t[i] = t; }
      }
      ++r;
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
    __syncthreads();
  }
  if (tid == 0) P.pf_count[b] = cap;
}

}  // namespace echo
