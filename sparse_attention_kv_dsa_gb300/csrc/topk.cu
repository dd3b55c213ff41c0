// Exact top-k with the EMA threshold update (sm_103a).
//
// "ECHO: Efficient KV Cache Offloading with Lossless Prefetching ..." review page:
//   "Problem and motivation" -- DSA keeps the 2048 highest-scoring tokens;
//   "Decode: predict the transfer, then recall exactly" -- the final selection is the
//   exact top-k, computed after the indexer;
//   "Key observations", Obs. 2 (Fig 7-8) -- the k-th score is tracked by an EMA with
//   smoothing 0.5, which is the next step's prefetch threshold.
//
// One thread-block cluster (8 CTAs x 512 threads, two CTAs per SM) per request; when the
// rows' clusters of 8 would not fit in one wave, the smallest cluster (1, 2 or 4 CTAs)
// whose slices still fit in shared memory.  Each CTA holds the
// order-preserving uint32 keys of a contiguous slice of the request's scores in
// shared memory.  A first pass histograms a window of keys around the key of the EMA
// threshold (the predicted k-th score; the window's width follows the last call's
// prediction error) and lists, per warp and in token order, every key from the window
// up; when the k-th key falls inside, one more pass over those lists finds the k-th
// largest key K* and the output is written from them, otherwise an MSB-first radix
// select over every key (11 + 11 + 10 bit digits) does.
// Each CTA histograms its slice and publishes the sums of its 32-bin groups; every CTA
// finds a digit from the group sums of all eight, then from the 32 bins of the chosen
// group, read through distributed shared memory, so every CTA derives the same digit
// with no broadcast step.  Output: every key > K*, then the tokens equal to
// K* with the lowest indices (ranks ordered across warps and CTAs), so ties go to
// the lower token index.  The selection order is ascending t within each class.
// echo_topk_prefetch also runs the indexer's deferred exact prefetch cap: after the
// last cluster barrier, the rank-0 CTA of a request whose qualifiers outnumber its
// cap reuses its shared memory for the fix-up (nothing to do in the common case).

#include <algorithm>
#include <cooperative_groups.h>

#include "common.cuh"
#include "pf_fixup.cuh"

namespace echo {

constexpr int TK_CL = 8;
constexpr int TK_THREADS = 512;         // two CTAs per SM: all clusters of a batch co-resident
constexpr int TK_WARPS = TK_THREADS / 32;
constexpr int TK_BINS = 2048;
constexpr int TK_BPT = TK_BINS / TK_THREADS;   // bins per thread (4)
constexpr int TK_KEYCAP = 23 * 1024;    // keys cached per CTA (92 KB)
static_assert(TK_THREADS == FX_THREADS, "the cap fix-up runs on one top-k CTA");

struct TkShared {
  uint32_t hist[2][TK_BINS];
  uint32_t warp_sums[32];
  uint32_t res[4];
  uint32_t cta_cnt[2];                  // [0] keys > K* (window pass: above the window, bit 31: a
                                        // warp's candidate list overflowed), [1] keys == K*
  uint32_t warp_gt[TK_WARPS], warp_eq[TK_WARPS];
  uint32_t warp_nl[TK_WARPS];           // candidate list lengths
  uint32_t coarse[2][TK_BINS / 32];     // sums of 32-bin groups of hist[buf] (read by the cluster)
  uint32_t tot_s[3];                    // window pass: keys above the window, in it, any overflow
  uint32_t minkey;
};
static_assert(TK_BPT == 4 && TK_THREADS == TK_BINS / 4, "eight threads sum one 32-bin group");

// This CTA's sums of 32-bin groups of its histogram h, for the other CTAs of the
// cluster.  Every thread calls it after h is complete; ends with a barrier.
__device__ __forceinline__ void tk_coarse(const uint32_t *h, uint32_t *coarse) {
  const int tid = threadIdx.x;
  const uint4 v = reinterpret_cast<const uint4 *>(h)[tid];   // bins 4 tid .. 4 tid + 3
  uint32_t s = v.x + v.y + v.z + v.w;
  s += __shfl_down_sync(0xffffffffu, s, 4);
  s += __shfl_down_sync(0xffffffffu, s, 2);
  s += __shfl_down_sync(0xffffffffu, s, 1);
  if ((tid & 7) == 0) coarse[tid >> 3] = s;
  __syncthreads();
}

// The bin, over the cluster's histograms h (and their group sums), that holds the
// need-th largest key counted from the top bin: res[0] = the bin, res[1] = keys in the
// bins above it.  Two small rounds of remote reads by one warp: the 64 group sums of
// every CTA, then the 32 bins of the chosen group.  Needs 1 <= need <= the keys in the
// histograms.  Every thread calls it after the cluster barrier that follows tk_coarse;
// ends with a barrier.
template <int CL>
__device__ __forceinline__ void tk_find(const uint32_t *h, const uint32_t *coarse, uint32_t need, uint32_t *res) {
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid < 32) {
    // lane L holds groups 63 - 2L (the higher) and 62 - 2L
    uint32_t a[CL], c[CL];
#pragma unroll
    for (uint32_t r = 0; r < CL; ++r) {
      a[r] = ld_dsmem_u32(map_dsmem(coarse + 63 - 2 * lane, r));
      c[r] = ld_dsmem_u32(map_dsmem(coarse + 62 - 2 * lane, r));
    }
    uint32_t hi = 0, lo = 0;
#pragma unroll
    for (uint32_t r = 0; r < CL; ++r) { hi += a[r]; lo += c[r]; }
    uint32_t incl = hi + lo;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += x;
    }
    const uint32_t ab = incl - hi - lo;                   // keys in the groups above both
    int g = -1;
    uint32_t gab = 0;
    if (ab < need && need <= ab + hi) { g = 63 - 2 * lane; gab = ab; }
    else if (ab + hi < need && need <= ab + hi + lo) { g = 62 - 2 * lane; gab = ab + hi; }
    const uint32_t m = __ballot_sync(0xffffffffu, g >= 0);
    const int src = m ? __ffs(m) - 1 : 0;
    g = max(__shfl_sync(0xffffffffu, g, src), 0);
    gab = __shfl_sync(0xffffffffu, gab, src);
    // lane i: bin 32 g + i
    uint32_t fv[CL];
#pragma unroll
    for (uint32_t r = 0; r < CL; ++r) fv[r] = ld_dsmem_u32(map_dsmem(h + 32 * g + lane, r));
    uint32_t f = 0;
#pragma unroll
    for (uint32_t r = 0; r < CL; ++r) f += fv[r];
    uint32_t sfx = f;                                      // bins 32 g + lane .. 32 g + 31
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_down_sync(0xffffffffu, sfx, o);
      if (lane + o < 32) sfx += x;
    }
    const uint32_t above = gab + sfx - f;
    if (above < need && need <= above + f) { res[0] = 32 * g + lane; res[1] = above; }
  }
  __syncthreads();
}

__device__ __forceinline__ float ema(float theta, float kth, float alpha) {
  if (isinf(kth) && kth < 0.f) return theta;                 // nothing selected
  if (isinf(theta) && theta > 0.f) return kth;               // first observation
  const float a = alpha, b = __fsub_rn(1.0f, alpha);
  return __fadd_rn(__fmul_rn(a, kth), __fmul_rn(b, theta));  // each op rounded, no FMA
}

// Relative error of the threshold as this step's prediction of the k-th score, for
// the adaptive prefetch cap: |theta - kth| / |kth|, 0 when either is not finite or
// kth = 0; written by the EMA's thread before it replaces theta.
__device__ __forceinline__ void record_pred_err(const PfFix &F, int b, float theta, float kth) {
  if (F.cap == nullptr || F.L.pf_pred_err == nullptr) return;
  const bool ok = isfinite(theta) && isfinite(kth) && kth != 0.f;
  F.L.pf_pred_err[b] = ok ? __fdiv_rn(fabsf(__fsub_rn(theta, kth)), fabsf(kth)) : 0.f;
}

template <int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(TK_THREADS, 2)
    topk_kernel(const float *scores, const int32_t *seq_len, int Lmax, int k, int32_t *out_idx, float *kth_out,
                float *theta, float alpha, int lcap, const __grid_constant__ PfFix F) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) unsigned char dsm[];
  TkShared &S = *reinterpret_cast<TkShared *>(dsm);
  uint32_t *keys = reinterpret_cast<uint32_t *>(dsm + ((sizeof(TkShared) + 15) & ~size_t(15)));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_rank();
  const int b = blockIdx.x / CL;
  const int L = min(max(seq_len[b], 0), Lmax);
  const float *sc = scores + (int64_t)b * Lmax;
  int32_t *out = out_idx + (int64_t)b * k;
  const int per = ((L + CL - 1) / CL + 3) & ~3;        // slice length, multiple of 4
  const int t0 = min(L, (int)rank * per), t1 = min(L, t0 + per);
  const int n = t1 - t0;
  // keys live in shared memory when the slice for Lmax fits (that is what was allocated)
  const int per_max = ((Lmax + CL - 1) / CL + 3) & ~3;
  const bool cached = per_max <= TK_KEYCAP;
  // per-warp candidate lists (token, key) after the keys: lcap entries per warp
  int32_t *list_t = reinterpret_cast<int32_t *>(keys + (cached ? per_max : 0));
  uint32_t *list_k = reinterpret_cast<uint32_t *>(list_t + TK_WARPS * lcap);
  // the threshold the indexer scored against, read before rank 0 updates it, and the
  // previous call's k-th score, read before rank 0 replaces it (it sizes the window)
  const float theta_scored = (F.cap != nullptr && rank == 0) ? theta[b] : 0.f;
  const float kth_hint = kth_out[b];

  if (L <= k) {
    // every token is selected; kth = smallest score
    uint32_t mn = 0xffffffffu;
    for (int i = tid; i < n; i += TK_THREADS) {
      out[t0 + i] = t0 + i;
      mn = min(mn, f32_key(sc[t0 + i]));
    }
    for (int i = L + (int)rank * TK_THREADS + tid; i < k; i += CL * TK_THREADS) out[i] = -1;
    mn = __reduce_min_sync(0xffffffffu, mn);
    if (tid == 0) S.minkey = 0xffffffffu;
    __syncthreads();
    if (lane == 0) atomicMin(&S.minkey, mn);
    __syncthreads();
    cluster_sync();
    if (rank == 0 && tid == 0) {
      uint32_t m = 0xffffffffu;
      for (uint32_t r = 0; r < CL; ++r) m = min(m, *cluster.map_shared_rank(&S.minkey, r));
      const float kv = L > 0 ? key_f32(m) : -INFINITY;
      kth_out[b] = kv;
      record_pred_err(F, b, theta[b], kv);
      theta[b] = ema(theta[b], kv, alpha);
    }
    cluster_sync();
    if (F.cap != nullptr && rank == 0) pf_fixup_block(F, b, theta_scored, *reinterpret_cast<PfFixSmem *>(dsm));
    return;
  }

  if (cached) {
    const float *src = sc + t0;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
      const int n4 = n >> 2;
      for (int i = tid; i < n4; i += TK_THREADS) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(src) + i);
        reinterpret_cast<uint4 *>(keys)[i] = make_uint4(f32_key(v.x), f32_key(v.y), f32_key(v.z), f32_key(v.w));
      }
      for (int i = 4 * n4 + tid; i < n; i += TK_THREADS) keys[i] = f32_key(src[i]);
    } else {
      for (int i = tid; i < n; i += TK_THREADS) keys[i] = f32_key(src[i]);
    }
  }
  __syncthreads();

  // ---- window pass around the predicted k-th key ----------------------------
  // The EMA threshold theta[b] predicts this step's k-th score.  One pass counts the
  // keys above a window of key values around it, histograms the window's keys in 2048
  // bins of 2^sb values, and lists every key from the window up (token, key) per warp,
  // in token order (warp w owns a contiguous part of the slice).  The window's half
  // width is 8x the distance between the prediction and the k-th key of the previous
  // call (left in kth_out, read before this call replaces it), a power of two from
  // 2^17 to 2^21 key values (2^21 without a finite previous key).  When the k-th key
  // falls in the window and no list overflowed, the last sb-bit pass and the output
  // read only the lists; otherwise the passes read every key.  Either way the result
  // is the exact k-th key: the width only decides how much work the lists save.
  const int wspan = (n + TK_WARPS - 1) / TK_WARPS;
  const int s0 = min(n, warp * wspan), s1 = min(n, s0 + wspan);
  uint32_t prefix = 0, above = 0;
  int left = 32, buf = 0;
  bool use_list = false;
  uint32_t nl = 0;                                         // this warp's list length
  const float th_pred = theta[b];
  int sb = 11;                                             // window bin width 2^sb
  if (isfinite(th_pred)) {                                // uniform across the cluster
    const uint32_t kt = f32_key(th_pred);
    if (isfinite(kth_hint)) {
      const uint32_t kp = f32_key(kth_hint);
      const uint64_t d8 = 8ull * (kt > kp ? kt - kp : kp - kt);
      sb = 7;
      while (sb < 11 && (1ull << (sb + 10)) < d8) ++sb;
    }
    const uint32_t half = 1u << (sb + 10);
    const uint32_t wlo = (kt > half ? kt - half : 0u) & ~((1u << sb) - 1u);
    const uint64_t whi = (uint64_t)wlo + 2ull * half;
    uint32_t *h = S.hist[0];
    for (int i = tid; i < TK_BINS; i += TK_THREADS) h[i] = 0;
    __syncthreads();
    uint32_t nab = 0, nwin = 0;
    int32_t *lt = list_t + warp * lcap;
    uint32_t *lk = list_k + warp * lcap;
    for (int i0 = s0; i0 < s1; i0 += 32) {                // warp-uniform trip count
      const int i = i0 + lane;
      uint32_t kk = 0;
      if (i < s1) kk = cached ? keys[i] : f32_key(sc[t0 + i]);
      const bool ab = i < s1 && (uint64_t)kk >= whi;
      const bool inw = i < s1 && kk >= wlo && (uint64_t)kk < whi;
      nab += ab ? 1u : 0u;                                 // per lane; summed over the warp below
      nwin += inw ? 1u : 0u;
      if (inw) atomicAdd(&h[(kk - wlo) >> sb], 1u);
      const uint32_t bal = __ballot_sync(0xffffffffu, ab || inw);
      if (ab || inw) {
        const uint32_t pos = nl + __popc(bal & lanemask_lt());
        if (pos < (uint32_t)lcap) {
          lt[pos] = t0 + i;
          lk[pos] = kk;
        }
      }
      nl += __popc(bal);
    }
    nab = __reduce_add_sync(0xffffffffu, nab);
    nwin = __reduce_add_sync(0xffffffffu, nwin);
    if (lane == 0) {
      S.warp_gt[warp] = nab;
      S.warp_eq[warp] = nwin;
      S.warp_nl[warp] = nl;
    }
    __syncthreads();
    if (tid == 0) {
      uint32_t t = 0, wn = 0, ovf = 0;
      for (int w = 0; w < TK_WARPS; ++w) {
        t += S.warp_gt[w];
        wn += S.warp_eq[w];
        ovf |= S.warp_nl[w] > (uint32_t)lcap ? 1u : 0u;
      }
      S.cta_cnt[0] = t | (ovf << 31);                      // counts stay below 2^31
      S.cta_cnt[1] = wn;
    }
    tk_coarse(h, S.coarse[0]);
    cluster_sync();
    // cluster totals: keys above the window, keys in it, any list overflow
    if (tid < 32) {
      const uint32_t ab = lane < CL ? ld_dsmem_u32(map_dsmem(&S.cta_cnt[0], lane)) : 0u;
      const uint32_t wn = lane < CL ? ld_dsmem_u32(map_dsmem(&S.cta_cnt[1], lane)) : 0u;
      const uint32_t tab_l = __reduce_add_sync(0xffffffffu, ab & 0x7fffffffu);
      const uint32_t tot_l = __reduce_add_sync(0xffffffffu, wn);
      const uint32_t ovf_l = __reduce_or_sync(0xffffffffu, ab >> 31);
      if (lane == 0) { S.tot_s[0] = tab_l; S.tot_s[1] = tot_l; S.tot_s[2] = ovf_l; }
    }
    __syncthreads();
    const uint32_t tab = S.tot_s[0], tot = S.tot_s[1], ovf = S.tot_s[2];
    if (tab < (uint32_t)k && (uint32_t)k <= tab + tot) {   // the k-th key is in the window
      tk_find<CL>(h, S.coarse[0], (uint32_t)k - tab, S.res);
      prefix = wlo + (S.res[0] << sb);
      above = tab + S.res[1];
      left = sb;
      use_list = lcap > 0 && ovf == 0;                     // uniform: every CTA read every flag
    }
    buf = 1;                        // other CTAs may still read hist[0]
    __syncthreads();
  }

  if (use_list) {
    // ---- last sb-bit pass over the lists: the keys of the chosen window bin ----
    uint32_t *h = S.hist[buf];
    for (int i = tid; i < TK_BINS; i += TK_THREADS) h[i] = 0;
    __syncthreads();
    const uint32_t *lk = list_k + warp * lcap;
    const int32_t *lt = list_t + warp * lcap;
    for (uint32_t j0 = 0; j0 < nl; j0 += 32) {              // warp-uniform trip count
      const uint32_t j = j0 + lane;
      const uint32_t kk = j < nl ? lk[j] : 0u;
      hist_add_warp(h, j < nl && (kk >> sb) == (prefix >> sb), kk & ((1u << sb) - 1u));   // one bin's keys: ties are common
    }
    __syncthreads();
    tk_coarse(h, S.coarse[buf]);
    cluster_sync();
    tk_find<CL>(h, S.coarse[buf], (uint32_t)k - above, S.res);
    prefix |= S.res[0];
    above += S.res[1];
    const uint32_t kstar = prefix;
    const uint32_t need_eq = (uint32_t)k - above;
    // ---- ordered output from the lists (every key >= K* is listed) ----
    uint32_t gt = 0, eq = 0;
    for (uint32_t j = lane; j < nl; j += 32) {
      const uint32_t kk = lk[j];
      gt += kk > kstar ? 1u : 0u;
      eq += kk == kstar ? 1u : 0u;
    }
    gt = __reduce_add_sync(0xffffffffu, gt);
    eq = __reduce_add_sync(0xffffffffu, eq);
    if (lane == 0) { S.warp_gt[warp] = gt; S.warp_eq[warp] = eq; }
    __syncthreads();
    if (tid == 0) {
      uint32_t a = 0, e = 0;
      for (int w = 0; w < TK_WARPS; ++w) {
        const uint32_t g = S.warp_gt[w], q = S.warp_eq[w];
        S.warp_gt[w] = a;
        S.warp_eq[w] = e;
        a += g;
        e += q;
      }
      S.cta_cnt[0] = a;
      S.cta_cnt[1] = e;
    }
    __syncthreads();
    cluster_sync();
    uint32_t gt_base = 0, eq_base = 0;
    {
      uint32_t g[CL], e[CL];
#pragma unroll
      for (uint32_t r = 0; r < CL; ++r) {
        g[r] = r < rank ? ld_dsmem_u32(map_dsmem(&S.cta_cnt[0], r)) : 0u;
        e[r] = r < rank ? ld_dsmem_u32(map_dsmem(&S.cta_cnt[1], r)) : 0u;
      }
#pragma unroll
      for (uint32_t r = 0; r < CL; ++r) { gt_base += g[r]; eq_base += e[r]; }
    }
    uint32_t gpos = gt_base + S.warp_gt[warp];
    uint32_t epos = eq_base + S.warp_eq[warp];
    for (uint32_t j0 = 0; j0 < nl; j0 += 32) {
      const uint32_t j = j0 + lane;
      const uint32_t kk = j < nl ? lk[j] : 0u;
      const bool isg = j < nl && kk > kstar, ise = j < nl && kk == kstar;
      const uint32_t bg = __ballot_sync(0xffffffffu, isg), be = __ballot_sync(0xffffffffu, ise);
      if (isg) out[gpos + __popc(bg & lanemask_lt())] = lt[j];
      if (ise) {
        const uint32_t er = epos + __popc(be & lanemask_lt());
        if (er < need_eq) out[above + er] = lt[j];
      }
      gpos += __popc(bg);
      epos += __popc(be);
    }
    if (rank == 0 && tid == 0) {
      const float kv = key_f32(kstar);
      kth_out[b] = kv;
      record_pred_err(F, b, theta[b], kv);
      theta[b] = ema(theta[b], kv, alpha);
    }
    cluster_sync();
    if (F.cap != nullptr && rank == 0) pf_fixup_block(F, b, theta_scored, *reinterpret_cast<PfFixSmem *>(dsm));
    return;
  }

  // ---- radix select of the k-th largest key -----------------------------
  while (left > 0) {
    const int w = min(11, left), shift = left - w;
    uint32_t *h = S.hist[buf];
    for (int i = tid; i < TK_BINS; i += TK_THREADS) h[i] = 0;
    __syncthreads();
    const uint32_t hi_mask = (shift + w >= 32) ? 0u : (0xffffffffu << (shift + w));
    for (int base = 0; base < n; base += TK_THREADS) {     // uniform trip count per warp
      const int i = base + tid;
      uint32_t kk = 0;
      if (i < n) kk = cached ? keys[i] : f32_key(sc[t0 + i]);
      if (i < n && (kk & hi_mask) == (prefix & hi_mask)) atomicAdd(&h[(kk >> shift) & ((1u << w) - 1)], 1u);
    }
    __syncthreads();
    tk_coarse(h, S.coarse[buf]);
    cluster_sync();
    tk_find<CL>(h, S.coarse[buf], (uint32_t)k - above, S.res);
    prefix |= S.res[0] << shift;
    above += S.res[1];
    left = shift;
    buf ^= 1;
    __syncthreads();
  }
  const uint32_t kstar = prefix;
  const uint32_t need_eq = (uint32_t)k - above;   // 1 <= need_eq <= count of keys == K*

  // ---- ordered output ---------------------------------------------------
  // warp w of this CTA owns the contiguous sub-range [s0, s1) of the slice
  uint32_t gt = 0, eq = 0;
  for (int i = s0 + lane; i < s1; i += 32) {
    const uint32_t kk = cached ? keys[i] : f32_key(sc[t0 + i]);
    gt += kk > kstar ? 1u : 0u;
    eq += kk == kstar ? 1u : 0u;
  }
  gt = __reduce_add_sync(0xffffffffu, gt);
  eq = __reduce_add_sync(0xffffffffu, eq);
  if (lane == 0) { S.warp_gt[warp] = gt; S.warp_eq[warp] = eq; }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0, e = 0;
    for (int w = 0; w < TK_WARPS; ++w) {
      const uint32_t g = S.warp_gt[w], q = S.warp_eq[w];
      S.warp_gt[w] = a;
      S.warp_eq[w] = e;
      a += g;
      e += q;
    }
    S.cta_cnt[0] = a;
    S.cta_cnt[1] = e;
  }
  __syncthreads();
  cluster_sync();
  uint32_t gt_base = 0, eq_base = 0;
  {
    uint32_t g[CL], e[CL];
#pragma unroll
    for (uint32_t r = 0; r < CL; ++r) {
      g[r] = r < rank ? ld_dsmem_u32(map_dsmem(&S.cta_cnt[0], r)) : 0u;
      e[r] = r < rank ? ld_dsmem_u32(map_dsmem(&S.cta_cnt[1], r)) : 0u;
    }
#pragma unroll
    for (uint32_t r = 0; r < CL; ++r) { gt_base += g[r]; eq_base += e[r]; }
  }
  uint32_t gpos = gt_base + S.warp_gt[warp];
  uint32_t epos = eq_base + S.warp_eq[warp];
  for (int i0 = s0; i0 < s1; i0 += 32) {
    const int i = i0 + lane;
    uint32_t kk = 0;
    if (i < s1) kk = cached ? keys[i] : f32_key(sc[t0 + i]);
    const bool isg = i < s1 && kk > kstar, ise = i < s1 && kk == kstar;
    const uint32_t bg = __ballot_sync(0xffffffffu, isg), be = __ballot_sync(0xffffffffu, ise);
    if (isg) out[gpos + __popc(bg & lanemask_lt())] = t0 + i;
    if (ise) {
      const uint32_t er = epos + __popc(be & lanemask_lt());
      if (er < need_eq) out[above + er] = t0 + i;
    }
    gpos += __popc(bg);
    epos += __popc(be);
  }
  if (rank == 0 && tid == 0) {
    const float kv = key_f32(kstar);
    kth_out[b] = kv;
    record_pred_err(F, b, theta[b], kv);
    theta[b] = ema(theta[b], kv, alpha);
  }
  cluster_sync();
  // no other CTA reads this one's shared memory any more: it becomes the fix-up's scratch
  if (F.cap != nullptr && rank == 0) pf_fixup_block(F, b, theta_scored, *reinterpret_cast<PfFixSmem *>(dsm));
}

// Entries per warp of the candidate lists: as many as fit (up to 256) while two CTAs
// still share an SM; 0 (no lists) when fewer than 64 fit.
static int topk_lcap(int Lmax, int cl) {
  static int per_sm = 0, reserved = 0;
  if (!per_sm) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (per_sm <= 0) per_sm = 1;
  }
  const int per = ((Lmax + cl - 1) / cl + 3) & ~3;
  const long base = (long)((sizeof(TkShared) + 15) & ~size_t(15)) + (per <= TK_KEYCAP ? (long)per * 4 : 0);
  const long room = (long)per_sm / 2 - reserved - base;
  if (room <= 0) return 0;
  const int lc = (int)std::min<long>(256, room / (TK_WARPS * 8)) & ~31;
  return lc >= 64 ? lc : 0;
}

static size_t topk_smem(int Lmax, int cl, int lcap, bool fix) {
  const int per = ((Lmax + cl - 1) / cl + 3) & ~3;
  size_t s = (sizeof(TkShared) + 15) & ~size_t(15);
  if (per <= TK_KEYCAP) s += (size_t)per * 4;
  s += (size_t)TK_WARPS * lcap * 8;
  if (fix) s = std::max(s, sizeof(PfFixSmem));
  return s;
}

template <int CL>
static echo_status_t run_topk(const float *scores, const int32_t *seq_len, int32_t B, int32_t Lmax, int32_t k,
                              int32_t *out_idx, float *kth, float *theta, float alpha, int lcap, size_t smem,
                              const PfFix &F, cudaStream_t st) {
  ECHO_CUDA_OK(cudaFuncSetAttribute(topk_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  topk_kernel<CL><<<B * CL, TK_THREADS, smem, st>>>(scores, seq_len, Lmax, k, out_idx, kth, theta, alpha, lcap, F);
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

static echo_status_t launch_topk(const float *scores, const int32_t *seq_len, int32_t B, int32_t Lmax, int32_t k,
                                 int32_t *out_idx, float *kth, float *theta, float alpha, const PfFix &F,
                                 echo_stream_t stream) {
  if (!scores || !seq_len || !out_idx || !kth || !theta || B <= 0 || Lmax <= 0 || k <= 0) return ECHO_ERR_INVALID_ARG;
  if (!(alpha >= 0.f && alpha <= 1.f)) return ECHO_ERR_INVALID_ARG;
  // A cluster of TK_CL CTAs per row while every row's cluster fits in one wave (two CTAs
  // per SM); with more rows, the smallest cluster whose slices still fit in shared
  // memory, so that short rows (blocks, many groups, prefill queries) take fewer CTAs.
  int cl = TK_CL;
  if ((int64_t)B * TK_CL > 2 * (int64_t)sm_count())
    for (cl = 1; cl < TK_CL && ((Lmax + cl - 1) / cl + 3) / 4 * 4 > TK_KEYCAP; cl *= 2) {
    }
  const int lcap = topk_lcap(Lmax, cl);
  const size_t smem = topk_smem(Lmax, cl, lcap, F.cap != nullptr);
  cudaStream_t st = (cudaStream_t)stream;
  switch (cl) {
    case 1: return run_topk<1>(scores, seq_len, B, Lmax, k, out_idx, kth, theta, alpha, lcap, smem, F, st);
    case 2: return run_topk<2>(scores, seq_len, B, Lmax, k, out_idx, kth, theta, alpha, lcap, smem, F, st);
    case 4: return run_topk<4>(scores, seq_len, B, Lmax, k, out_idx, kth, theta, alpha, lcap, smem, F, st);
    default: return run_topk<TK_CL>(scores, seq_len, B, Lmax, k, out_idx, kth, theta, alpha, lcap, smem, F, st);
  }
}

}  // namespace echo

using namespace echo;

extern "C" echo_status_t echo_topk(const float *scores, const int32_t *seq_len, int32_t B, int32_t Lmax, int32_t k,
                                   int32_t *out_idx, float *kth, float *theta, float alpha, echo_stream_t stream) {
  const PfFix none = {};
  return launch_topk(scores, seq_len, B, Lmax, k, out_idx, kth, theta, alpha, none, stream);
}

extern "C" echo_status_t echo_topk_prefetch(const float *scores, const int32_t *seq_len, int32_t B, int32_t Lmax,
                                            int32_t k, int32_t *out_idx, float *kth, float *theta, float alpha,
                                            const int32_t *cap, int32_t cap_max, const int32_t *host_base,
                                            const echo_cache_layer_t *layer, int32_t *pf_list, int32_t *pf_count,
                                            void *stage_kv, echo_stream_t stream) {
  if (!cap || cap_max <= 0 || !host_base || !layer || !pf_list || !pf_count || !stage_kv) return ECHO_ERR_INVALID_ARG;
  if (!layer->host2gpu || !layer->host_kv) return ECHO_ERR_INVALID_ARG;
  if (!layer_takes_prefetch(layer)) return ECHO_ERR_UNSUPPORTED;
  const PfFix F = {seq_len, Lmax, cap, cap_max, host_base, *layer, scores, pf_list, pf_count, stage_kv};
  return launch_topk(scores, seq_len, B, Lmax, k, out_idx, kth, theta, alpha, F, stream);
}
