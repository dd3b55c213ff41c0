// Lightning-indexer scoring with fused threshold prefetch (sm_103a).
//
// "ECHO: Efficient KV Cache Offloading with Lossless Prefetching ..." review page:
//   "Problem and motivation"  -- the DSA lightning indexer scores every past token
//                                (score(t) = sum_h w_h * ReLU(q_h . k_t), DeepSeek-V3.2-Exp
//                                report in the show notes' sources); top-2048 follows.
//   "Decode: predict the transfer, then recall exactly" -- the EMA of the 2048-th
//                                score is the prefetch threshold; once a block of scores
//                                exists, tokens above it that are not cached are fetched
//                                without waiting for the top-k; a counter caps the volume.
//   "Fusing prefetch into the indexer pipeline" -- prefetch overlaps the scoring stream.
//
// FP8 kernel (H = 64 heads, D = 128): persistent CTAs, two per SM (two independent
// pipelines per SM measured 1.5x faster than one CTA with deeper rings), each walking
// a contiguous range of the 128-token tiles of all requests.  Warp roles:
//   warp 0     TMA producer: 16 KB key tiles (128 tokens x 128 B, 128-byte swizzle)
//              through a 4-stage mbarrier ring, plus the request's q (64 x 128 B)
//   warp 1     one thread issues tcgen05.mma kind::f8f6f4, M=128 tokens, N=64 heads,
//              K=128 (4 x 32), accumulating in TMEM (4 x 64 columns)
//   warp 2     prefetch: residency check, capped claim, zero-copy copy of the latent
//              row from pinned host memory into the request's staging rows
//   warps 3-6  epilogue: tcgen05.ld of a token row (64 head dot products), ReLU,
//              weighted sum (packed fma.rn.f32x2, two heads per instruction), score
//              store; tokens above the threshold go to a ring
// On the exact grid the tensor-core sums are exact, so scores equal the definition.
// The cap is exact: claims are optimistic (any order) and a fix-up restores "the first
// cap tokens by ascending t" for the rare request whose qualifiers outnumber its cap,
// either in its own small launch here or, deferred, inside the top-k kernel.

#include <algorithm>
#include <cstddef>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "pf_fixup.cuh"

namespace echo {

constexpr int IX_TILE = 128;
constexpr int IX_H = 64;
constexpr int IX_D = 128;
#ifndef ECHO_IX_STAGES
#define ECHO_IX_STAGES 4          // key tiles in flight per CTA
#endif
#ifndef ECHO_IX_CTAS_PER_SM
#define ECHO_IX_CTAS_PER_SM 2     // persistent CTAs per SM (two independent pipelines)
#endif
#ifndef ECHO_IX_EPI_GROUPS
#define ECHO_IX_EPI_GROUPS 1      // epilogue warp groups (4 warps each) taking tiles in turn
#endif
#ifndef ECHO_IX_MMA_GROUP
#define ECHO_IX_MMA_GROUP 1       // tiles whose MMAs are interleaved
#endif
#ifndef ECHO_IX_WB
#define ECHO_IX_WB 16             // requests whose head weights are kept in shared memory
#endif
constexpr int IX_STAGES = ECHO_IX_STAGES;
constexpr int IX_RING = 1024;
constexpr int IX_MAXB = 1024;
constexpr int IX_EPI = ECHO_IX_EPI_GROUPS;
constexpr int IX_MMA_GROUP = ECHO_IX_MMA_GROUP;
static_assert(IX_MMA_GROUP <= 2, "two q buffers: at most one deferred release per group");
constexpr int IX_THREADS = (3 + 4 * IX_EPI) * 32;   // producer, MMA, prefetch, epilogue groups
constexpr int IX_KTILE_BYTES = IX_TILE * IX_D;   // 16384
constexpr int IX_Q_BYTES = IX_H * IX_D;          // 8192
constexpr int IX_ACC = 4;                        // TMEM accumulator buffers (4 x 64 columns)
constexpr int IX_WB = ECHO_IX_WB;


struct IxParams {
  const float *w;
  const int32_t *seq_len;
  int B, Lmax;
  const float *theta;
  const int32_t *cap;       // null: no prefetch
  int cap_max;
  const int32_t *host_base;
  echo_cache_layer_t L;
  float *scores;
  int32_t *pf_list;
  int32_t *pf_count;
  void *stage_kv;
};

struct IxSmemTail {
  uint64_t full[IX_STAGES], empty[IX_STAGES];
  uint64_t qfull[2], qempty[2], tfull[IX_ACC], tempty[IX_ACC];
  uint32_t tmem_base;
  uint32_t ring_tail;
  uint32_t ring_head;
  uint32_t ring_claim;
  uint32_t epi_done;
  int32_t tile_pre[IX_MAXB + 1];
  int32_t ring_b[IX_RING];
  int32_t ring_t[IX_RING];
  int32_t ring_seq[IX_RING];
  alignas(16) float w_s[IX_WB * IX_H];            // head weights of the first IX_WB requests (float4 reads)
  float theta_s[IX_MAXB];
  int32_t len_s[IX_MAXB];
};

static_assert(offsetof(IxSmemTail, w_s) % 16 == 0, "float4 reads of the head weights need 16-byte alignment");
static_assert((IX_STAGES * IX_KTILE_BYTES + 2 * IX_Q_BYTES) % 1024 == 0, "tail must start 1024-byte aligned");
constexpr size_t IX_SMEM = 1024 /*align slack*/ + IX_STAGES * IX_KTILE_BYTES + 2 * IX_Q_BYTES + sizeof(IxSmemTail);

__device__ __forceinline__ int find_req(const int32_t *pre, int B, int tile) {
  int lo = 0, hi = B - 1;  // last b with pre[b] <= tile
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= tile) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Claim staging rows for the qualifying lanes of a warp and copy their latent rows.
// Every lane passes (valid, b, t, h); returns nothing.  Used by the prefetch warp.
__device__ __forceinline__ void claim_and_copy(const IxParams &P, bool cand, int b, int t) {
  const echo_cache_layer_t &L = P.L;
  bool qual = false;
  int64_t h = 0;
  if (cand) {
    h = (int64_t)P.host_base[b] + t;
    if (h < 0 || h >= L.n_host) {
      set_status(L.counters, ECHO_ERR_HOST_INDEX);
    } else {
      qual = L.host2gpu[h] == -1;
    }
  }
  int32_t row = -1;
  if (qual) {
    const int cap = min(P.cap[b], P.cap_max);
    const int pos = atomicAdd(&P.pf_count[b], 1);
    if (pos < cap) {
      row = b * P.cap_max + pos;
      P.pf_list[row] = t;
      P.L.host2gpu[h] = -2 - row;
    }
  }
  const uint32_t nq = __popc(__ballot_sync(0xffffffffu, qual));
  uint32_t mk = __ballot_sync(0xffffffffu, row >= 0);
  if ((threadIdx.x & 31) == 0) {
    if (nq) atomicAdd(&L.counters[ECHO_CTR_QUALIFIED], (int)nq);
    if (mk) atomicAdd(&L.counters[ECHO_CTR_STAGED], __popc(mk));
  }
  const int esz = L.kv_dtype == ECHO_F32 ? 4 : 2;
  const int chunks = KV_W * esz / 16;
  while (mk) {
    const uint4 *src[4] = {nullptr, nullptr, nullptr, nullptr};
    uint4 *dst[4] = {nullptr, nullptr, nullptr, nullptr};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (!mk) break;
      const int ln = __ffs(mk) - 1;
      mk &= mk - 1;
      const int64_t hh = __shfl_sync(0xffffffffu, h, ln);
      const int32_t rr = __shfl_sync(0xffffffffu, row, ln);
      src[j] = reinterpret_cast<const uint4 *>((const char *)L.host_kv + hh * KV_W * esz);
      dst[j] = reinterpret_cast<uint4 *>((char *)P.stage_kv + (int64_t)rr * KV_W * esz);
    }
    warp_copy_rows4(src, dst, chunks);
  }
}

// One consumer step on the candidate ring: claim up to 32 entries (CAS on the claim
// cursor), read them, process them (residency check, capped claim, copy).
// Returns false when nothing was available.  Whole warp.
__device__ __forceinline__ bool consume_ring(const IxParams &P, IxSmemTail &S, int32_t *ctr) {
  const int lane = threadIdx.x & 31;
  uint32_t c = 0, n = 0;
  if (lane == 0) {
    while (true) {
      c = *(volatile uint32_t *)&S.ring_claim;
      const uint32_t tail = *(volatile uint32_t *)&S.ring_tail;
      if (c >= tail) { n = 0; break; }
      n = min(tail - c, 32u);
      if (atomicCAS(&S.ring_claim, c, c + n) == c) break;
    }
  }
  c = __shfl_sync(0xffffffffu, c, 0);
  n = __shfl_sync(0xffffffffu, n, 0);
  if (n == 0) return false;
  bool cand = false;
  int b = 0, t = 0;
  if ((uint32_t)lane < n) {
    const uint32_t pos = c + lane;
    const int slot = pos % IX_RING;
    const uint64_t tw = global_ns();
    bool ok = true;
    while (*(volatile int32_t *)&S.ring_seq[slot] != (int32_t)(pos + 1)) {
      if (global_ns() - tw > kWaitLimitNs) { ok = false; break; }
    }
    __threadfence_block();
    b = S.ring_b[slot];
    t = S.ring_t[slot];
    cand = ok && b >= 0;
    if (!ok) set_status(ctr, ECHO_ERR_TIMEOUT);
  }
  __syncwarp();
  if (lane == 0) atomicAdd(&S.ring_head, n);         // entries read: ring space for producers
  claim_and_copy(P, cand, b, t);
  return true;
}

__global__ void __launch_bounds__(IX_THREADS, ECHO_IX_CTAS_PER_SM)
    indexer_fp8_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                       IxParams P) {
  extern __shared__ unsigned char dsm_raw[];
  unsigned char *dsm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
  unsigned char *kbuf = dsm;
  unsigned char *qbuf = dsm + IX_STAGES * IX_KTILE_BYTES;
  IxSmemTail &S = *reinterpret_cast<IxSmemTail *>(qbuf + 2 * IX_Q_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool prefetch = P.cap != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < IX_STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.qfull[s], 1);
      mbar_init(&S.qempty[s], 1);
    }
    for (int s = 0; s < IX_ACC; ++s) {
      mbar_init(&S.tfull[s], 1);
      mbar_init(&S.tempty[s], 128);
    }
    S.ring_tail = 0;
    S.ring_head = 0;
    S.ring_claim = 0;
    S.epi_done = 0;
    fence_mbar_init();
  }
  block_prefix(P.B, [&](int b) { return (min(max(P.seq_len[b], 0), P.Lmax) + IX_TILE - 1) / IX_TILE; },
               S.tile_pre);
  for (int i = threadIdx.x; i < IX_RING; i += IX_THREADS) S.ring_seq[i] = 0;
  for (int i = threadIdx.x; i < min(P.B, IX_WB) * IX_H; i += IX_THREADS) S.w_s[i] = P.w[i];
  for (int i = threadIdx.x; i < P.B; i += IX_THREADS) {
    S.theta_s[i] = P.theta[i];
    S.len_s[i] = min(P.seq_len[i], P.Lmax);
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, IX_ACC * IX_H);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int T = S.tile_pre[P.B];
  // this CTA's contiguous range of tiles [i0, i1): a CTA meets few requests, so it
  // rarely reloads a query block or head weights (both stall the pipeline)
  const int i0 = (int)(((int64_t)T * blockIdx.x) / gridDim.x);
  const int i1 = (int)(((int64_t)T * (blockIdx.x + 1)) / gridDim.x);
  const uint32_t tmem = S.tmem_base;
  int32_t *ctr = P.L.counters;

  if (warp == 0) {
    // ---------------------------------------------------------- producer --
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&qmap);
      const uint64_t stream_once = l2_evict_first_policy();   // keys are read once per step
      int it = 0, qn = 0, cur = -1;
      for (int i = i0; i < i1; ++i, ++it) {
        const int b = find_req(S.tile_pre, P.B, i);
        const int t0 = (i - S.tile_pre[b]) * IX_TILE;
        if (b != cur) {
          const int qs = qn & 1;
          if (!mbar_wait(&S.qempty[qs], ((qn >> 1) & 1) ^ 1)) { set_status(ctr, ECHO_ERR_TIMEOUT); break; }
          mbar_arrive_expect_tx(&S.qfull[qs], IX_Q_BYTES);
          tma_load_2d(qbuf + qs * IX_Q_BYTES, &qmap, &S.qfull[qs], 0, b * IX_H);
          ++qn;
          cur = b;
        }
        const int s = it % IX_STAGES;
        const uint32_t ph = (it / IX_STAGES) & 1;
        if (!mbar_wait(&S.empty[s], ph ^ 1)) { set_status(ctr, ECHO_ERR_TIMEOUT); break; }
        mbar_arrive_expect_tx(&S.full[s], IX_KTILE_BYTES);
        tma_load_2d_hint(kbuf + s * IX_KTILE_BYTES, &kmap, &S.full[s], 0, b * P.Lmax + t0, stream_once);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA --
    // Tiles are issued in groups of IX_MMA_GROUP with their K-steps interleaved, so
    // consecutive MMAs target different accumulators and the tensor pipe can overlap
    // them (the four K-steps of one tile depend on each other).
    if (lane == 0) {
      constexpr uint32_t idesc = instr_desc(FMT_E4M3, FMT_E4M3, 0, 0, IX_TILE, IX_H);
      int it = 0, qn = 0, cur = -1, qs = 0;
      bool ok = true;
      for (int i = i0; i < i1 && ok;) {
        int st[IX_MMA_GROUP], ac[IX_MMA_GROUP], qsl[IX_MMA_GROUP];
        int n = 0, defer = -1;
        for (; n < IX_MMA_GROUP && i < i1; ++n, ++it, ++i) {
          const int b = find_req(S.tile_pre, P.B, i);
          if (b != cur) {
            if (cur >= 0) {
              // release the previous request's q buffer once no pending MMA reads it
              if (n > 0) defer = qs; else mma_commit(&S.qempty[qs]);
            }
            qs = qn & 1;
            if (!mbar_wait(&S.qfull[qs], (qn >> 1) & 1)) { ok = false; break; }
            ++qn;
            cur = b;
          }
          st[n] = it % IX_STAGES;
          ac[n] = it % IX_ACC;
          qsl[n] = qs;
          if (!mbar_wait(&S.tempty[ac[n]], ((it / IX_ACC) & 1) ^ 1) ||
              !mbar_wait(&S.full[st[n]], (it / IX_STAGES) & 1)) { ok = false; break; }
        }
        if (!ok) { set_status(ctr, ECHO_ERR_TIMEOUT); break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < IX_D / 32; ++kk)
          for (int j = 0; j < n; ++j) {
            const uint64_t ad = smem_desc(smem_u32(kbuf + st[j] * IX_KTILE_BYTES), 16, 1024, LAYOUT_SW128);
            const uint64_t bd = smem_desc(smem_u32(qbuf + qsl[j] * IX_Q_BYTES), 16, 1024, LAYOUT_SW128);
            mma_f8f6f4(tmem + ac[j] * IX_H, ad + 2 * kk, bd + 2 * kk, idesc, kk > 0 ? 1u : 0u);
          }
        for (int j = 0; j < n; ++j) {
          mma_commit(&S.empty[st[j]]);
          mma_commit(&S.tfull[ac[j]]);
        }
        if (defer >= 0) mma_commit(&S.qempty[defer]);
      }
    }
  } else if (warp >= 3) {
    // ---------------------------------------------------------- epilogue --
    // group g (4 warps, one per TMEM lane quadrant) takes the tiles with it % IX_EPI == g
    const int grp = (warp - 3) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    float wr[IX_H];
    float theta = 0.f;
    int Lb = 0, cur = -1;
    int it = 0;
    for (int i = i0; i < i1; ++i, ++it) {
      if (it % IX_EPI != grp) continue;
      const int b = find_req(S.tile_pre, P.B, i);
      const int t0 = (i - S.tile_pre[b]) * IX_TILE;
      if (b != cur) {
        const float4 *wp = reinterpret_cast<const float4 *>(b < IX_WB ? S.w_s + b * IX_H : P.w + (int64_t)b * IX_H);
#pragma unroll
        for (int j = 0; j < IX_H / 4; ++j) {
          const float4 v = wp[j];
          wr[4 * j] = v.x; wr[4 * j + 1] = v.y; wr[4 * j + 2] = v.z; wr[4 * j + 3] = v.w;
        }
        theta = S.theta_s[b];
        Lb = S.len_s[b];
        cur = b;
      }
      const int acc = it % IX_ACC;
      if (!mbar_wait(&S.tfull[acc], (it / IX_ACC) & 1)) { set_status(ctr, ECHO_ERR_TIMEOUT); break; }
      tc_fence_after();
      uint32_t r0[32], r1[32];
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + acc * IX_H;
      tmem_ld32(taddr, r0);
      tmem_ld32(taddr + 32, r1);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&S.tempty[acc]);
      // eight independent partial sums in four packed pairs (every partial sum is exact
      // on the grid); one fma.rn.f32x2 per pair of heads
      unsigned long long c[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int p = 0; p < 32; ++p) {
        const uint32_t *rr = p < 16 ? r0 : r1;
        const int hh = 2 * (p & 15);
        unsigned long long xv, wv;
        asm("mov.b64 %0, {%1, %2};" : "=l"(xv) : "f"(fmaxf(__uint_as_float(rr[hh]), 0.f)),
            "f"(fmaxf(__uint_as_float(rr[hh + 1]), 0.f)));
        asm("mov.b64 %0, {%1, %2};" : "=l"(wv) : "f"(wr[2 * p]), "f"(wr[2 * p + 1]));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(c[p & 3]) : "l"(wv), "l"(xv));
      }
      float e[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) asm("mov.b64 {%0, %1}, %2;" : "=f"(e[2 * q]), "=f"(e[2 * q + 1]) : "l"(c[q]));
      const float sc = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
      const int t = t0 + row;
      if (t < Lb) {
        P.scores[(int64_t)b * P.Lmax + t] = sc;
        if (prefetch && sc > theta) {
          const uint32_t pos = atomicAdd(&S.ring_tail, 1u);
          bool ok = true;
          if ((int)(pos - *(volatile uint32_t *)&S.ring_head) >= IX_RING) {   // ring full: bounded wait
            const uint64_t tw = global_ns();
            while ((int)(pos - *(volatile uint32_t *)&S.ring_head) >= IX_RING) {
              if (global_ns() - tw > kWaitLimitNs) { ok = false; break; }
              __nanosleep(64);
            }
          }
          const int slot = pos % IX_RING;
          S.ring_b[slot] = ok ? b : -1;
          S.ring_t[slot] = t;
          __threadfence_block();
          *(volatile int32_t *)&S.ring_seq[slot] = (int32_t)(pos + 1);
          if (!ok) set_status(ctr, ECHO_ERR_TIMEOUT);
        }
      }
    }
    __threadfence_block();
    atomicAdd(&S.epi_done, 1u);
    if (prefetch) {
      // once every epilogue thread is done (no more pushes), help drain the ring
      const uint64_t tw = global_ns();
      while (*(volatile uint32_t *)&S.epi_done < 128u * IX_EPI) {
        if (global_ns() - tw > kWaitLimitNs) { set_status(ctr, ECHO_ERR_TIMEOUT); break; }
        __nanosleep(128);
      }
      __threadfence_block();
      while (consume_ring(P, S, ctr)) {
      }
    }
  } else if (warp == 2 && prefetch) {
    // ---------------------------------------------------------- prefetch --
    uint64_t t_idle = global_ns();
    while (true) {
      const uint32_t done = *(volatile uint32_t *)&S.epi_done;
      __threadfence_block();
      if (consume_ring(P, S, ctr)) {
        t_idle = global_ns();
        continue;
      }
      if (done == 128u * IX_EPI) break;                // all pushed and all claimed
      if (global_ns() - t_idle > 4 * kWaitLimitNs) { set_status(ctr, ECHO_ERR_TIMEOUT); break; }
      __nanosleep(256);                                // idle: leave the issue slots to the epilogue
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, IX_ACC * IX_H);
}

// ------------------------------------------------------- float32 SIMT path --
// One thread per token; q of the request in shared memory.  For the float32
// workload (few heads, short context); same prefetch rule, inline claim and copy.
constexpr int SX_THREADS = 128;
__global__ void __launch_bounds__(SX_THREADS)
    indexer_f32_kernel(const float *q, const float *keys, int H, int D, IxParams P) {
  extern __shared__ float qs[];
  const int b = blockIdx.y;
  const int L = min(P.seq_len[b], P.Lmax);
  const int t0 = blockIdx.x * SX_THREADS;
  if (t0 >= L) return;
  for (int i = threadIdx.x; i < H * D; i += SX_THREADS) qs[i] = q[(int64_t)b * H * D + i];
  __syncthreads();
  const int t = t0 + threadIdx.x;
  bool cand = false;
  if (t < L) {
    const float4 *kr = reinterpret_cast<const float4 *>(keys + ((int64_t)b * P.Lmax + t) * D);
    float sc = 0.f;
    for (int h = 0; h < H; ++h) {
      float d = 0.f;
      const float4 *qh = reinterpret_cast<const float4 *>(qs + h * D);
      for (int j = 0; j < D / 4; ++j) {
        const float4 kv = __ldg(kr + j), qv = qh[j];
        d = fmaf(qv.x, kv.x, d);
        d = fmaf(qv.y, kv.y, d);
        d = fmaf(qv.z, kv.z, d);
        d = fmaf(qv.w, kv.w, d);
      }
      sc = fmaf(P.w[(int64_t)b * H + h], fmaxf(d, 0.f), sc);
    }
    P.scores[(int64_t)b * P.Lmax + t] = sc;
    cand = P.cap != nullptr && sc > P.theta[b];
  }
  if (P.cap != nullptr && __any_sync(0xffffffffu, cand)) claim_and_copy(P, cand, b, t);
}

// --------------------------------------------------- exact cap, rare path --
__global__ void __launch_bounds__(FX_THREADS) pf_finalize_kernel(const __grid_constant__ PfFix F, const float *theta) {
  __shared__ PfFixSmem sm;
  pf_fixup_block(F, blockIdx.x, theta[blockIdx.x], sm);
}

// ------------------------------------------------------------- host side --
static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D byte tensor [rows, 128] with a [box_rows, 128] box and 128-byte swizzle.
bool make_map_128B(CUtensorMap *m, const void *base, uint64_t rows, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace echo

using namespace echo;

extern "C" echo_status_t echo_index_prefetch(const void *q, const float *w, const void *idx_k,
                                             const int32_t *seq_len, int32_t B, int32_t H, int32_t D,
                                             int32_t Lmax, int32_t dtype, const float *theta, const int32_t *cap,
                                             int32_t cap_max, const int32_t *host_base,
                                             const echo_cache_layer_t *layer, float *scores, int32_t *pf_list,
                                             int32_t *pf_count, void *stage_kv, int32_t flags,
                                             echo_stream_t stream) {
  if (!q || !w || !idx_k || !seq_len || !theta || !scores || B <= 0 || B > IX_MAXB || Lmax <= 0)
    return ECHO_ERR_INVALID_ARG;
  if (flags & ~ECHO_PF_DEFER_CAP) return ECHO_ERR_INVALID_ARG;
  if (cap) {
    if (!layer || !host_base || !pf_list || !pf_count || !stage_kv || cap_max <= 0) return ECHO_ERR_INVALID_ARG;
    if (!layer->host2gpu || !layer->host_kv || !layer->counters) return ECHO_ERR_INVALID_ARG;
    if (!layer_takes_prefetch(layer)) return ECHO_ERR_UNSUPPORTED;
  }
  IxParams P = {};
  P.w = w;
  P.seq_len = seq_len;
  P.B = B;
  P.Lmax = Lmax;
  P.theta = theta;
  P.cap = cap;
  P.cap_max = cap_max;
  P.host_base = host_base;
  if (layer) P.L = *layer;
  P.scores = scores;
  P.pf_list = pf_list;
  P.pf_count = pf_count;
  P.stage_kv = stage_kv;
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == ECHO_E4M3) {
    if (H != IX_H || D != IX_D) return ECHO_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(idx_k) | reinterpret_cast<uintptr_t>(q)) & 15) return ECHO_ERR_INVALID_ARG;
    CUtensorMap kmap, qmap;
    if (!make_map_128B(&kmap, idx_k, (uint64_t)B * Lmax, IX_TILE)) return ECHO_ERR_CUDA;
    if (!make_map_128B(&qmap, q, (uint64_t)B * IX_H, IX_H)) return ECHO_ERR_CUDA;
    ECHO_CUDA_OK(cudaFuncSetAttribute(indexer_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)IX_SMEM));
    const int64_t tmax = (int64_t)B * ((Lmax + IX_TILE - 1) / IX_TILE);
    const int grid = (int)std::min<int64_t>((int64_t)sm_count() * ECHO_IX_CTAS_PER_SM, tmax);
    indexer_fp8_kernel<<<grid, IX_THREADS, IX_SMEM, st>>>(kmap, qmap, P);
    ECHO_LAUNCH_OK();
  } else if (dtype == ECHO_F32) {
    if (H <= 0 || D <= 0 || D % 4 != 0 || H * D > 8192) return ECHO_ERR_UNSUPPORTED;
    dim3 grid((Lmax + SX_THREADS - 1) / SX_THREADS, B);
    indexer_f32_kernel<<<grid, SX_THREADS, H * D * sizeof(float), st>>>((const float *)q, (const float *)idx_k, H,
                                                                         D, P);
    ECHO_LAUNCH_OK();
  } else {
    return ECHO_ERR_UNSUPPORTED;
  }
  if (cap && !(flags & ECHO_PF_DEFER_CAP)) {
    const PfFix F = {seq_len, Lmax, cap, cap_max, host_base, P.L, scores, pf_list, pf_count, stage_kv};
    pf_finalize_kernel<<<B, FX_THREADS, 0, st>>>(F, theta);
    ECHO_LAUNCH_OK();
  }
  return ECHO_OK;
}
