// Prefill chunk indexing with coarse-histogram candidates (sm_103a).
//
// "ECHO: Efficient KV Cache Offloading with Lossless Prefetching ..." review page,
// "Prefill: overlap recall across query blocks": a prefill chunk is scored in query
// blocks; while block i+1 is scored, the KV of the candidates already identified for
// block i is transferred.  Instead of a full top-k inside the scoring pipeline, a
// 256-bucket coarse histogram picks the buckets that are certainly above the
// selection boundary and leaves the threshold bucket for later; subtracting the
// predicted k-th score first makes the buckets near the boundary finer.  The exact
// top-k and recall follow ("Decode: predict the transfer, then recall exactly").
//
// Kernels
//   prefill_score_kernel  tcgen05: one 128-token key tile (A, M = 128) against four
//                         queries' 64 heads (B, N = 256), K = 128, FP8 e4m3 with f32
//                         accumulators in TMEM (two 256-column buffers).  The epilogue
//                         forms sum_h w_h ReLU(.) per (token, query), stores the causal
//                         scores and histograms bucket(score - kth_pred) per query.
//                         Persistent CTAs walk contiguous runs of (query quad, range of
//                         key tiles) items.
//                         Warp 0 TMA producer, warp 1 MMA issuer, warps 2-9 epilogue (two
//                         warps per TMEM lane quadrant, two queries each).
//   prefill_cand_kernel   one CTA per query: threshold bucket from the histogram,
//                         then a pass over the query's scores marking the tokens of
//                         higher buckets in a token bitmap (one OR per warp and word).
//   mark_kernel           marks rows of token lists (the exact selections) in a bitmap.
//   token_list_kernel     bitmap -> ascending token list (padded with -1), clears it.

#include <algorithm>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace echo {

constexpr int PF_TILE = 128;                     // tokens per key tile (MMA M)
constexpr int PF_H = 64;                         // indexer heads
constexpr int PF_D = 128;                        // indexer dim (bytes per e4m3 row)
constexpr int PF_QG = 4;                         // queries per MMA (N = 4 x 64)
constexpr int PF_N = PF_QG * PF_H;               // 256
constexpr int PF_STAGES = 4;                     // key tiles in flight
constexpr int PF_ACC = 2;                        // TMEM accumulators of 256 columns
constexpr int PF_RANGE = 64;                     // key tiles per work item
constexpr int PF_EPI = 256;                       // epilogue threads: two warps per TMEM lane quadrant
constexpr int PF_THREADS = 64 + PF_EPI;           // producer, MMA, 8 epilogue warps
constexpr int PF_KTILE_BYTES = PF_TILE * PF_D;   // 16 KB
constexpr int PF_Q_BYTES = PF_N * PF_D;          // 32 KB
constexpr int PF_BUCKETS = 256;

struct PfParams {
  const float *w;          // [Q, 64]
  const float *kth_pred;   // [Q]
  int Q, Lmax, pos0;
  int ntiles, nrange, nitems;
  float *scores;           // [Q, Lmax]
  uint32_t *hist;          // [Q, 256]
  int32_t *status;         // optional
};

struct PfSmemTail {
  uint64_t full[PF_STAGES], empty[PF_STAGES];
  uint64_t qfull[2], qempty[2], tfull[PF_ACC], tempty[PF_ACC];
  uint32_t tmem_base;
  alignas(16) float w_s[PF_QG * PF_H];
  float kth_s[PF_QG];
  uint32_t hist_s[PF_QG * PF_BUCKETS];
};
static_assert((PF_STAGES * PF_KTILE_BYTES + 2 * PF_Q_BYTES) % 1024 == 0, "tail must start 1024-byte aligned");
constexpr size_t PF_SMEM = 1024 + PF_STAGES * PF_KTILE_BYTES + 2 * PF_Q_BYTES + sizeof(PfSmemTail);

__device__ __forceinline__ void pf_status(int32_t *st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}
// Named barrier of the epilogue threads (barrier 1; barrier 0 is __syncthreads).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(PF_EPI) : "memory"); }

// Tiles [ja, jb) of work item i: query quad g, key-tile range r; tiles past the
// quad's last causal position are skipped.
struct PfItem {
  int g, ja, jb;
};
__device__ __forceinline__ PfItem pf_item(const PfParams &P, int i) {
  PfItem it;
  it.g = i / P.nrange;
  const int r = i % P.nrange;
  const int last_q = min(P.Q, PF_QG * it.g + PF_QG) - 1;            // last query of the quad
  const int nt = (P.pos0 + last_q) / PF_TILE + 1;                     // tiles up to its position
  it.ja = r * PF_RANGE;
  it.jb = min(min(nt, P.ntiles), it.ja + PF_RANGE);
  return it;
}

// Order-preserving uint32 key of a float (larger float -> larger key; -0 == +0).
__device__ __forceinline__ uint32_t pf_key(float x) { return f32_key(x); }

__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_score_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                         PfParams P) {
  extern __shared__ unsigned char pf_raw[];
  unsigned char *dsm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(pf_raw) + 1023) & ~uintptr_t(1023));
  unsigned char *kbuf = dsm;
  unsigned char *qbuf = dsm + PF_STAGES * PF_KTILE_BYTES;
  PfSmemTail &S = *reinterpret_cast<PfSmemTail *>(qbuf + 2 * PF_Q_BYTES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < PF_STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.qfull[s], 1);
      mbar_init(&S.qempty[s], 1);
    }
    for (int s = 0; s < PF_ACC; ++s) {
      mbar_init(&S.tfull[s], 1);
      mbar_init(&S.tempty[s], PF_EPI);
    }
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < PF_QG * PF_BUCKETS; i += PF_THREADS) S.hist_s[i] = 0;
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, PF_ACC * PF_N);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  // this CTA's contiguous range of items [i0, i1): consecutive items share a query quad,
  // so its queries, weights and histograms change rarely
  const int i0 = (int)(((int64_t)P.nitems * blockIdx.x) / gridDim.x);
  const int i1 = (int)(((int64_t)P.nitems * (blockIdx.x + 1)) / gridDim.x);

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&qmap);
      int it = 0, qn = 0, cur = -1;
      bool ok = true;
      for (int i = i0; i < i1 && ok; ++i) {
        const PfItem w = pf_item(P, i);
        if (w.ja >= w.jb) continue;
        if (w.g != cur) {
          const int qs = qn & 1;
          if (!mbar_wait(&S.qempty[qs], ((qn >> 1) & 1) ^ 1)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.qfull[qs], PF_Q_BYTES);
          tma_load_2d(qbuf + qs * PF_Q_BYTES, &qmap, &S.qfull[qs], 0, w.g * PF_N);
          ++qn;
          cur = w.g;
        }
        for (int j = w.ja; j < w.jb; ++j, ++it) {
          const int s = it % PF_STAGES;
          if (!mbar_wait(&S.empty[s], ((it / PF_STAGES) & 1) ^ 1)) { ok = false; break; }
          mbar_arrive_expect_tx(&S.full[s], PF_KTILE_BYTES);
          tma_load_2d(kbuf + s * PF_KTILE_BYTES, &kmap, &S.full[s], 0, j * PF_TILE);
        }
      }
      if (!ok) pf_status(P.status, ECHO_ERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA --
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc(FMT_E4M3, FMT_E4M3, 0, 0, PF_TILE, PF_N);
      int it = 0, qn = 0, cur = -1, qs = 0;
      bool ok = true;
      for (int i = i0; i < i1 && ok; ++i) {
        const PfItem w = pf_item(P, i);
        if (w.ja >= w.jb) continue;
        if (w.g != cur) {
          if (cur >= 0) mma_commit(&S.qempty[qs]);       // previous quad's MMAs are all issued
          qs = qn & 1;
          if (!mbar_wait(&S.qfull[qs], (qn >> 1) & 1)) { ok = false; break; }
          ++qn;
          cur = w.g;
        }
        for (int j = w.ja; j < w.jb; ++j, ++it) {
          const int s = it % PF_STAGES, acc = it % PF_ACC;
          if (!mbar_wait(&S.tempty[acc], ((it / PF_ACC) & 1) ^ 1) ||
              !mbar_wait(&S.full[s], (it / PF_STAGES) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = smem_desc(smem_u32(kbuf + s * PF_KTILE_BYTES), 16, 1024, LAYOUT_SW128);
          const uint64_t bd = smem_desc(smem_u32(qbuf + qs * PF_Q_BYTES), 16, 1024, LAYOUT_SW128);
#pragma unroll
          for (int kk = 0; kk < PF_D / 32; ++kk)
            mma_f8f6f4(tmem + acc * PF_N, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0 ? 1u : 0u);
          mma_commit(&S.empty[s]);
          mma_commit(&S.tfull[acc]);
        }
      }
      if (!ok) pf_status(P.status, ECHO_ERR_TIMEOUT);
    }
  } else {
    // ---------------------------------------------------------- epilogue --
    const int quad = warp & 3;                         // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;                  // token within the tile
    const int et = threadIdx.x - 64;                   // 0..PF_EPI-1
    const int qh = (warp - 2) >> 2;                    // which two of the quad's four queries
    int it = 0, cur = -1;
    bool ok = true;
    // adds the quad's histograms into the global ones and clears them
    auto flush = [&](int g) {
      epi_sync();
      for (int i = et; i < PF_QG * PF_BUCKETS; i += PF_EPI) {
        const uint32_t v = S.hist_s[i];
        const int q = PF_QG * g + i / PF_BUCKETS;
        if (v && q < P.Q) atomicAdd(&P.hist[(int64_t)q * PF_BUCKETS + (i % PF_BUCKETS)], v);
        S.hist_s[i] = 0;
      }
      epi_sync();
    };
    // every epilogue warp walks every item (the named barriers need all four), even
    // after a bounded wait gave up (its tiles are then skipped)
    for (int i = i0; i < i1; ++i) {
      const PfItem w = pf_item(P, i);
      if (w.ja >= w.jb) continue;
      if (w.g != cur) {
        if (cur >= 0) flush(cur);
        for (int x = et; x < PF_QG * PF_H; x += PF_EPI) {
          const int q = PF_QG * w.g + x / PF_H;
          S.w_s[x] = q < P.Q ? P.w[(int64_t)q * PF_H + (x % PF_H)] : 0.f;
        }
        if (et < PF_QG) {
          const int q = PF_QG * w.g + et;
          S.kth_s[et] = q < P.Q ? P.kth_pred[q] : 0.f;
        }
        epi_sync();
        cur = w.g;
      }
      for (int j = w.ja; j < w.jb && ok; ++j, ++it) {
        const int acc = it % PF_ACC;
        if (!mbar_wait(&S.tfull[acc], (it / PF_ACC) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + acc * PF_N;
        const int t = j * PF_TILE + row;
        float sc[2];
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int qi = 2 * qh + qq;
          uint32_t r0[32], r1[32];
          tmem_ld32(taddr + qi * PF_H, r0);
          tmem_ld32(taddr + qi * PF_H + 32, r1);
          tmem_wait_ld();
          const float *wq = S.w_s + qi * PF_H;
          // four independent partial sums (each exact on the synthetic grid)
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
          for (int h = 0; h < 32; h += 2) {
            a0 = fmaf(wq[h], fmaxf(__uint_as_float(r0[h]), 0.f), a0);
            a1 = fmaf(wq[h + 1], fmaxf(__uint_as_float(r0[h + 1]), 0.f), a1);
            a2 = fmaf(wq[32 + h], fmaxf(__uint_as_float(r1[h]), 0.f), a2);
            a3 = fmaf(wq[33 + h], fmaxf(__uint_as_float(r1[h + 1]), 0.f), a3);
          }
          sc[qq] = (a0 + a1) + (a2 + a3);
        }
        tc_fence_before();
        mbar_arrive(&S.tempty[acc]);
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
          const int qi = 2 * qh + qq;
          const int q = PF_QG * w.g + qi;
          if (q < P.Q && t <= P.pos0 + q && t < P.Lmax) {      // causal range of query q
            P.scores[(int64_t)q * P.Lmax + t] = sc[qq];
            const uint32_t bkt = pf_key(__fsub_rn(sc[qq], S.kth_s[qi])) >> 24;
            atomicAdd(&S.hist_s[qi * PF_BUCKETS + bkt], 1u);
          }
        }
      }
    }
    if (cur >= 0) flush(cur);
    if (!ok) pf_status(P.status, ECHO_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, PF_ACC * PF_N);
}

// ------------------------------------------------------------- candidates --
constexpr int PC_THREADS = 512;

__global__ void __launch_bounds__(PC_THREADS)
    prefill_cand_kernel(const float *scores, const uint32_t *hist, int Q, int Lmax, int pos0, int k,
                        const float *kth_pred, int32_t *thr_out, int32_t *cand_count, uint32_t *bitmap) {
  __shared__ int32_t pre[PF_BUCKETS + 1];
  __shared__ int32_t thr_s;
  __shared__ uint32_t wcnt[PC_THREADS / 32];
  const int q = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Lq = min(pos0 + q + 1, Lmax);
  // threshold bucket: the bucket holding the k-th largest (counts from bucket 255 down)
  block_prefix(PF_BUCKETS, [&](int i) { return (int)hist[(int64_t)q * PF_BUCKETS + (PF_BUCKETS - 1 - i)]; }, pre);
  if (tid == 0) thr_s = -1;
  __syncthreads();
  if (Lq > k && tid < PF_BUCKETS && pre[tid] < k && pre[tid + 1] >= k) thr_s = PF_BUCKETS - 1 - tid;
  __syncthreads();
  const int thr = thr_s;
  const float kth = kth_pred[q];
  const float *sc = scores + (int64_t)q * Lmax;
  uint32_t n = 0;
  for (int base = 0; base < Lq; base += PC_THREADS) {        // warps cover 32 aligned tokens
    const int t = base + tid;
    const bool c = t < Lq && (int)(f32_key(__fsub_rn(__ldg(sc + t), kth)) >> 24) > thr;
    const uint32_t bal = __ballot_sync(0xffffffffu, c);
    if (lane == 0 && bal) atomicOr(&bitmap[t >> 5], bal);
    n += __popc(bal);
  }
  if (lane == 0) wcnt[warp] = n;
  __syncthreads();
  if (tid == 0) {
    uint32_t tot = 0;
    for (int w = 0; w < PC_THREADS / 32; ++w) tot += wcnt[w];
    if (cand_count) cand_count[q] = (int32_t)tot;
    if (thr_out) thr_out[q] = thr;
  }
}

// ------------------------------------------------------ bitmap <-> lists --
__global__ void mark_kernel(const int32_t *tok, int64_t n, uint32_t *bitmap, int nbits) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t t = tok[i];
    if (t >= 0 && t < nbits) atomicOr(&bitmap[t >> 5], 1u << (t & 31));
  }
}

constexpr int TL_THREADS = 1024;

__global__ void __launch_bounds__(TL_THREADS)
    token_list_kernel(uint32_t *bitmap, int nbits, int32_t *list, int cap, int32_t *count) {
  __shared__ int32_t pre[TL_THREADS + 1];
  const int tid = threadIdx.x;
  const int nw = (nbits + 31) >> 5;
  const int per = (nw + TL_THREADS - 1) / TL_THREADS;
  const int w0 = min(nw, tid * per), w1 = min(nw, w0 + per);
  int c = 0;
  for (int w = w0; w < w1; ++w) c += __popc(bitmap[w]);
  block_prefix(TL_THREADS, [&](int) { return c; }, pre);     // f(i) is evaluated by thread i
  int pos = pre[tid];
  for (int w = w0; w < w1; ++w) {
    uint32_t m = bitmap[w];
    bitmap[w] = 0;                                          // left clear for the next use
    while (m) {
      const int b = __ffs(m) - 1;
      m &= m - 1;
      if (pos < cap) list[pos] = (w << 5) + b;
      ++pos;
    }
  }
  const int total = pre[TL_THREADS];
  for (int i = total + tid; i < cap; i += TL_THREADS) list[i] = -1;
  if (tid == 0) *count = total;
}

// Slot of every listed token (prefill attention): one thread per entry.
__global__ void translate_kernel(echo_cache_layer_t L, const int32_t *tok, int64_t n, int k,
                                 const int32_t *host_base, int per_row, int32_t *out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t t = tok[i];
    int32_t g = -1;
    if (t >= 0) {
      const int64_t h = (int64_t)host_base[per_row ? i / k : 0] + t;
      if (h < 0 || h >= L.n_host) {
        set_status(L.counters, ECHO_ERR_HOST_INDEX);
      } else {
        g = L.host2gpu[h];
        if (g < 0) {                                 // not resident (or staged in a step)
          set_status(L.counters, ECHO_ERR_NOT_RESIDENT);
          g = -1;
        }
      }
    }
    out[i] = g;
  }
}

}  // namespace echo

using namespace echo;

extern "C" echo_status_t echo_prefill_index(const void *q, const float *w, const void *idx_k, int32_t Q, int32_t H,
                                            int32_t D, int32_t Lmax, int32_t pos0, const float *kth_pred,
                                            float *scores, uint32_t *hist, int32_t *status, echo_stream_t stream) {
  if (!q || !w || !idx_k || !kth_pred || !scores || !hist || Q <= 0 || Lmax <= 0 || pos0 < 0)
    return ECHO_ERR_INVALID_ARG;
  if ((int64_t)pos0 + Q > Lmax) return ECHO_ERR_INVALID_ARG;      // every query's own key is in the cache
  if (H != PF_H || D != PF_D) return ECHO_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(idx_k)) & 15) return ECHO_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  ECHO_CUDA_OK(cudaMemsetAsync(hist, 0, sizeof(uint32_t) * PF_BUCKETS * (size_t)Q, st));
  CUtensorMap kmap, qmap;
  if (!make_map_128B(&kmap, idx_k, (uint64_t)Lmax, PF_TILE)) return ECHO_ERR_CUDA;
  if (!make_map_128B(&qmap, q, (uint64_t)Q * PF_H, PF_N)) return ECHO_ERR_CUDA;
  PfParams P = {};
  P.w = w;
  P.kth_pred = kth_pred;
  P.Q = Q;
  P.Lmax = Lmax;
  P.pos0 = pos0;
  P.ntiles = (pos0 + Q + PF_TILE - 1) / PF_TILE;
  P.nrange = (P.ntiles + PF_RANGE - 1) / PF_RANGE;
  P.nitems = ((Q + PF_QG - 1) / PF_QG) * P.nrange;
  P.scores = scores;
  P.hist = hist;
  P.status = status;
  ECHO_CUDA_OK(cudaFuncSetAttribute(prefill_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PF_SMEM));
  const int grid = std::min(sm_count(), P.nitems);
  prefill_score_kernel<<<grid, PF_THREADS, PF_SMEM, st>>>(kmap, qmap, P);
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

extern "C" echo_status_t echo_prefill_candidates(const float *scores, const uint32_t *hist, int32_t Q, int32_t Lmax,
                                                 int32_t pos0, int32_t k, const float *kth_pred, int32_t *thr,
                                                 int32_t *cand_count, uint32_t *bitmap, echo_stream_t stream) {
  if (!scores || !hist || !kth_pred || !bitmap || Q <= 0 || Lmax <= 0 || pos0 < 0 || k <= 0)
    return ECHO_ERR_INVALID_ARG;
  prefill_cand_kernel<<<Q, PC_THREADS, 0, (cudaStream_t)stream>>>(scores, hist, Q, Lmax, pos0, k, kth_pred, thr,
                                                                   cand_count, bitmap);
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

extern "C" echo_status_t echo_mark_tokens(const int32_t *tok, int32_t rows, int32_t row_len, uint32_t *bitmap,
                                          int32_t nbits, echo_stream_t stream) {
  if (!tok || !bitmap || rows <= 0 || row_len <= 0 || nbits <= 0) return ECHO_ERR_INVALID_ARG;
  const int64_t n = (int64_t)rows * row_len;
  const int grid = (int)std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 8);
  mark_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(tok, n, bitmap, nbits);
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

extern "C" echo_status_t echo_token_list(uint32_t *bitmap, int32_t nbits, int32_t *list, int32_t cap,
                                         int32_t *count, echo_stream_t stream) {
  if (!bitmap || !list || !count || nbits <= 0 || cap <= 0) return ECHO_ERR_INVALID_ARG;
  token_list_kernel<<<1, TL_THREADS, 0, (cudaStream_t)stream>>>(bitmap, nbits, list, cap, count);
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

extern "C" echo_status_t echo_translate_slots(const echo_cache_layer_t *layer, const int32_t *tok, int32_t rows,
                                              int32_t k, const int32_t *host_base, int32_t per_row_base,
                                              int32_t *out_slot, echo_stream_t stream) {
  if (!layer || !tok || !host_base || !out_slot || rows <= 0 || k <= 0) return ECHO_ERR_INVALID_ARG;
  if (!layer->host2gpu || !layer->counters || layer->n_host <= 0) return ECHO_ERR_INVALID_ARG;
  const int64_t n = (int64_t)rows * k;
  const int grid = (int)std::min<int64_t>((n + 255) / 256, (int64_t)sm_count() * 8);
  translate_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(*layer, tok, n, k, host_base, per_row_base != 0,
                                                           out_slot);
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}
