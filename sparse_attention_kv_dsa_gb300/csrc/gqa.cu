// Sparse attention of a GQA layer with several KV heads (N4).
//
// "ECHO: Efficient KV Cache Offloading with Lossless Prefetching ..." review page,
// critique section: the design adapts to GQA models by adding a KV-head dimension to
// its cache.  Each (request, KV head) pair -- a group -- has its own selection of
// token rows; a row holds the token's key (d values) then its value (d values).  The
// group's G query heads attend over its rows:
//   logit_j = scale * q_g . key_j,  out_g = softmax_j(logit) . value_j,  lse_g = log sum_j exp(logit_j).
//
// bf16 path: one CTA per (group, split of 256 selected rows), four warps.  Rows are
// gathered by cp.async into a two-stage ring of 64-row tiles (keys and values in
// 128-byte-swizzled shared memory).  Each warp owns 16 rows of a tile: S = Q K^T and
// O += P V run on the warp-level bf16 tensor-core MMA (m16n8k16, f32 accumulate) with
// the G <= 16 query heads as the M dimension, with an online softmax in base 2.  The
// four warps' states are merged in shared memory; several splits are merged by a
// combine kernel.  The work is a gather: about 8 flops per byte of rows, so HBM and the
// gather's latency bound it, not the tensor rate -- the warp-level MMA covers it with
// G as small as 8 (the 5th-generation MMA's smallest M is 64).
// f32 path: the same splits and merge on CUDA cores (exact float32 arithmetic).

#include <algorithm>
#include <cmath>

#include "common.cuh"

namespace echo {

constexpr int GQ_THREADS = 128;   // four warps
constexpr int GQ_TS = 256;        // selected rows per split (CTA)
constexpr int GQ_CH = 64;         // rows per pipeline tile (16 per warp)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct GqaPart {
  float *o;    // [NG, ns, G, d]  sum_j 2^(s_j - m) value_j
  float *ml;   // [NG, ns, G, 2]  (m, l), base-2 units of the scaled logits
};

static int gqa_splits(int k) { return (k + GQ_TS - 1) / GQ_TS; }

// ------------------------------------------------------ warp-level MMA helpers --
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// c += a (16x16, row) * b (16x8, col), bf16 inputs, f32 accumulate
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Shared-memory tile of rows x (D values) bf16: 16-byte chunk c of row r is stored at
// chunk (c ^ (r & 7)), so eight rows read at the same chunk hit eight bank groups.
template <int D>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int r, int c) {
  return base + (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// ------------------------------------------------------------------ bf16 split --
template <int D>
__global__ void __launch_bounds__(GQ_THREADS) gqa_bf16_kernel(const __nv_bfloat16 *__restrict__ q,
                                                              const __nv_bfloat16 *__restrict__ kv, int kv_rows,
                                                              const int32_t *__restrict__ slot_idx, int G, int k,
                                                              int ns, float scale_log2, GqaPart part,
                                                              __nv_bfloat16 *__restrict__ out, float *__restrict__ lse) {
  constexpr int KC = D / 8;                              // 16-byte chunks per key (or value)
  constexpr int TILE = GQ_CH * D * 2;                    // bytes of one 64-row key (or value) tile
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *stage = smem;                           // [2][K tile, V tile]
  unsigned char *qs = smem + 4 * TILE;                   // Q tile [16][D] bf16
  int32_t *s_slot = reinterpret_cast<int32_t *>(qs + 16 * D * 2);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = blockIdx.x / ns, sp = blockIdx.x % ns;
  const int j0 = sp * GQ_TS, nrow = min(GQ_TS, k - j0);
  const int nch = (nrow + GQ_CH - 1) / GQ_CH;

  for (int j = tid; j < GQ_TS; j += GQ_THREADS) {
    int32_t g = j < nrow ? slot_idx[(int64_t)n * k + j0 + j] : -1;
    s_slot[j] = (g >= 0 && g < kv_rows) ? g : -1;
  }
  // Q rows G..15 are zero
  for (int i = tid; i < 16 * KC; i += GQ_THREADS) {
    const int r = i / KC, c = i % KC;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < G) v = reinterpret_cast<const uint4 *>(q + ((int64_t)n * G + r) * D)[c];
    *reinterpret_cast<uint4 *>(qs + (r * (D * 2) + ((c ^ (r & 7)) << 4))) = v;
  }
  __syncthreads();

  auto load_tile = [&](int c, int buf) {
    unsigned char *kt = stage + buf * 2 * TILE, *vt = kt + TILE;
    for (int i = tid; i < GQ_CH * 2 * KC; i += GQ_THREADS) {
      const int r = i / (2 * KC), cc = i % (2 * KC);
      const int32_t g = s_slot[c * GQ_CH + r];
      const __nv_bfloat16 *src = kv + (g >= 0 ? (int64_t)g * 2 * D : 0) + cc * 8;
      unsigned char *t = cc < KC ? kt : vt;
      const int ch = cc < KC ? cc : cc - KC;
      cp_async_16(t + r * (D * 2) + ((ch ^ (r & 7)) << 4), src, g >= 0 ? 16u : 0u);
    }
  };
  if (nch > 0) load_tile(0, 0);
  cp_async_commit();
  if (nch > 1) load_tile(1, 1);
  cp_async_commit();

  // A fragments of Q (rows = query heads, k = d)
  uint32_t qa[D / 16][4];
  {
    const int mi = lane >> 3, r = (mi & 1) * 8 + (lane & 7);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) ldsm_x4(tile_addr<D>(smem_u32(qs), r, ks * 2 + (mi >> 1)), qa[ks]);
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows gid and gid + 8
  const int tig = lane & 3;

  for (int c = 0; c < nch; ++c) {
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t kt = smem_u32(stage + (c & 1) * 2 * TILE), vt = kt + TILE;
    const int rw = warp * 16;                             // this warp's 16 rows of the tile
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, r = rw + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t b[4];
        ldsm_x4(tile_addr<D>(kt, r, ks * 2 + (mi & 1)), b);
        mma_16816(s[0], qa[ks], b[0], b[1]);
        mma_16816(s[1], qa[ks], b[2], b[3]);
      }
    }
    // mask, scale (base 2), online softmax
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool ok = s_slot[c * GQ_CH + rw + t * 8 + 2 * tig + e] >= 0;
        s[t][e] = ok ? s[t][e] * scale_log2 : -INFINITY;
        s[t][2 + e] = ok ? s[t][2 + e] * scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, s[t][e]);
        mx1 = fmaxf(mx1, s[t][2 + e]);
      }
#pragma unroll
    for (int x = 1; x <= 2; x <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
    }
    const float n0 = fmaxf(m0, mx0), n1 = fmaxf(m1, mx1);
    const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
    const float c0 = exp2f(m0 - u0), c1 = exp2f(m1 - u1);
    m0 = n0;
    m1 = n1;
    float p[2][4];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      p[t][0] = exp2f(s[t][0] - u0);
      p[t][1] = exp2f(s[t][1] - u0);
      p[t][2] = exp2f(s[t][2] - u1);
      p[t][3] = exp2f(s[t][3] - u1);
    }
    l0 = l0 * c0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
    l1 = l1 * c1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= c0;
      o[i][1] *= c0;
      o[i][2] *= c1;
      o[i][3] *= c1;
    }
    const uint32_t pa[4] = {pack_bf16(p[0][0], p[0][1]), pack_bf16(p[0][2], p[0][3]), pack_bf16(p[1][0], p[1][1]),
                            pack_bf16(p[1][2], p[1][3])};
    {
      const int mi = lane >> 3, r = rw + (mi & 1) * 8 + (lane & 7);
#pragma unroll
      for (int jd = 0; jd < D / 16; ++jd) {
        uint32_t b[4];
        ldsm_x4_t(tile_addr<D>(vt, r, jd * 2 + (mi >> 1)), b);
        mma_16816(o[2 * jd], pa, b[0], b[1]);
        mma_16816(o[2 * jd + 1], pa, b[2], b[3]);
      }
    }
    __syncthreads();                                      // every warp is done with this buffer
    if (c + 2 < nch) load_tile(c + 2, c & 1);
    cp_async_commit();
  }
  cp_async_wait_all();
  __syncthreads();

  // merge the four warps (the ring's memory is free now)
#pragma unroll
  for (int x = 1; x <= 2; x <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, x);
    l1 += __shfl_xor_sync(0xffffffffu, l1, x);
  }
  float *ow = reinterpret_cast<float *>(stage);           // [4][16][D]
  float *mw = ow + 4 * 16 * D, *lw = mw + 4 * 16;          // [4][16]
  const int gid = lane >> 2;
#pragma unroll
  for (int i = 0; i < D / 8; ++i) {
    const int col = i * 8 + 2 * tig;
    *reinterpret_cast<float2 *>(ow + (warp * 16 + gid) * D + col) = make_float2(o[i][0], o[i][1]);
    *reinterpret_cast<float2 *>(ow + (warp * 16 + gid + 8) * D + col) = make_float2(o[i][2], o[i][3]);
  }
  if (tig == 0) {
    mw[warp * 16 + gid] = m0;
    mw[warp * 16 + gid + 8] = m1;
    lw[warp * 16 + gid] = l0;
    lw[warp * 16 + gid + 8] = l1;
  }
  __syncthreads();
  for (int i = tid; i < G * D; i += GQ_THREADS) {
    const int r = i / D, e = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * 16 + r]);
    float O = 0.f, Lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float f = exp2f(mw[w * 16 + r] - M);
        O += f * ow[(w * 16 + r) * D + e];
        Lsum += f * lw[w * 16 + r];
      }
    }
    if (ns == 1) {
      out[((int64_t)n * G + r) * D + e] = __float2bfloat16(Lsum > 0.f ? O / Lsum : 0.f);
      if (e == 0) lse[(int64_t)n * G + r] = Lsum > 0.f ? (M + log2f(Lsum)) * kLn2 : -INFINITY;
    } else {
      const int64_t row = ((int64_t)n * ns + sp) * G + r;
      part.o[row * D + e] = O;
      if (e == 0) {
        part.ml[row * 2] = M;
        part.ml[row * 2 + 1] = Lsum;
      }
    }
  }
}

// ------------------------------------------------------------------- f32 split --
template <int D>
__global__ void __launch_bounds__(GQ_THREADS) gqa_f32_kernel(const float *__restrict__ q, const float *__restrict__ kv,
                                                             int kv_rows, const int32_t *__restrict__ slot_idx, int G,
                                                             int k, int ns, float scale, GqaPart part,
                                                             float *__restrict__ out, float *__restrict__ lse) {
  constexpr int PL = D / 32;                             // values per lane
  __shared__ int32_t s_slot[GQ_TS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = blockIdx.x / ns, sp = blockIdx.x % ns;
  const int j0 = sp * GQ_TS, nrow = min(GQ_TS, k - j0);
  for (int j = tid; j < GQ_TS; j += GQ_THREADS) {
    int32_t g = j < nrow ? slot_idx[(int64_t)n * k + j0 + j] : -1;
    s_slot[j] = (g >= 0 && g < kv_rows) ? g : -1;
  }
  __syncthreads();
  for (int h = warp; h < G; h += GQ_THREADS / 32) {
    float qv[PL], ov[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) {
      qv[i] = q[((int64_t)n * G + h) * D + lane + 32 * i];
      ov[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < nrow; ++j) {
      const int32_t g = s_slot[j];
      if (g < 0) continue;
      const float *row = kv + (int64_t)g * 2 * D;
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < PL; ++i) dot = fmaf(qv[i], row[lane + 32 * i], dot);
#pragma unroll
      for (int x = 16; x > 0; x >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, x);
      const float logit = dot * scale;
      const float mn = fmaxf(m, logit);
      const float corr = expf(m - mn), p = expf(logit - mn);
      l = l * corr + p;
#pragma unroll
      for (int i = 0; i < PL; ++i) ov[i] = ov[i] * corr + p * row[D + lane + 32 * i];
      m = mn;
    }
    if (ns == 1) {
#pragma unroll
      for (int i = 0; i < PL; ++i) out[((int64_t)n * G + h) * D + lane + 32 * i] = l > 0.f ? ov[i] / l : 0.f;
      if (lane == 0) lse[(int64_t)n * G + h] = l > 0.f ? m + logf(l) : -INFINITY;
    } else {
      const int64_t row = ((int64_t)n * ns + sp) * G + h;
#pragma unroll
      for (int i = 0; i < PL; ++i) part.o[row * D + lane + 32 * i] = ov[i];
      if (lane == 0) {                                   // the merge works in base 2
        part.ml[row * 2] = m == -INFINITY ? m : m * kLog2e;
        part.ml[row * 2 + 1] = l;
      }
    }
  }
}

// ---------------------------------------------------------------- split merge --
template <typename OutT>
__global__ void gqa_combine_kernel(GqaPart part, int ns, int G, int D, OutT *__restrict__ out,
                                   float *__restrict__ lse) {
  const int r = blockIdx.x, n = blockIdx.y;                // query head, group
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, part.ml[(((int64_t)n * ns + s) * G + r) * 2]);
  float L = 0.f;
  if (M != -INFINITY)
    for (int s = 0; s < ns; ++s) {
      const int64_t row = ((int64_t)n * ns + s) * G + r;
      L += exp2f(part.ml[row * 2] - M) * part.ml[row * 2 + 1];
    }
  for (int e = threadIdx.x; e < D; e += blockDim.x) {
    float O = 0.f;
    if (M != -INFINITY)
      for (int s = 0; s < ns; ++s) {
        const int64_t row = ((int64_t)n * ns + s) * G + r;
        O += exp2f(part.ml[row * 2] - M) * part.o[row * D + e];
      }
    const float v = L > 0.f ? O / L : 0.f;
    if constexpr (sizeof(OutT) == 2)
      out[((int64_t)n * G + r) * D + e] = __float2bfloat16(v);
    else
      out[((int64_t)n * G + r) * D + e] = v;
  }
  if (threadIdx.x == 0) lse[(int64_t)n * G + r] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

template <int D>
static constexpr size_t gqa_bf16_smem() {
  return 4 * (size_t)GQ_CH * D * 2 + 16 * D * 2 + GQ_TS * 4;
}

template <int D>
static echo_status_t launch_gqa(const void *q, const void *kv, int kv_rows, int dtype, const int32_t *slot_idx,
                                int NG, int G, int k, float scale, void *out, float *lse, GqaPart part, int ns,
                                cudaStream_t st) {
  const unsigned grid = (unsigned)NG * (unsigned)ns;
  if (dtype == ECHO_BF16) {
    constexpr size_t smem = gqa_bf16_smem<D>();
    static_assert(4 * 16 * D * 4 + 2 * 4 * 16 * 4 <= 4 * GQ_CH * D * 2, "merge area fits in the ring");
    ECHO_CUDA_OK(cudaFuncSetAttribute(gqa_bf16_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    gqa_bf16_kernel<D><<<grid, GQ_THREADS, smem, st>>>((const __nv_bfloat16 *)q, (const __nv_bfloat16 *)kv, kv_rows,
                                                       slot_idx, G, k, ns, scale * kLog2e, part,
                                                       (__nv_bfloat16 *)out, lse);
    ECHO_LAUNCH_OK();
    if (ns > 1) gqa_combine_kernel<__nv_bfloat16><<<dim3(G, NG), 128, 0, st>>>(part, ns, G, D, (__nv_bfloat16 *)out, lse);
  } else {
    gqa_f32_kernel<D><<<grid, GQ_THREADS, 0, st>>>((const float *)q, (const float *)kv, kv_rows, slot_idx, G, k, ns,
                                                   scale, part, (float *)out, lse);
    ECHO_LAUNCH_OK();
    if (ns > 1) gqa_combine_kernel<float><<<dim3(G, NG), 128, 0, st>>>(part, ns, G, D, (float *)out, lse);
  }
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

}  // namespace echo

using namespace echo;

extern "C" size_t echo_sparse_gqa_workspace_bytes(int32_t NG, int32_t G, int32_t d, int32_t k) {
  if (NG <= 0 || G <= 0 || d <= 0 || k <= 0) return 0;
  const int ns = gqa_splits(k);
  return ns > 1 ? (size_t)NG * ns * G * (d + 2) * sizeof(float) : 0;
}

extern "C" echo_status_t echo_sparse_gqa_decode(const void *q, const void *kv, int32_t kv_rows, int32_t dtype,
                                                const int32_t *slot_idx, int32_t NG, int32_t G, int32_t d, int32_t k,
                                                float scale, void *out, float *lse, void *workspace,
                                                size_t workspace_bytes, echo_stream_t stream) {
  if (!q || !kv || !slot_idx || !out || !lse || NG <= 0 || G <= 0 || k <= 0 || kv_rows <= 0)
    return ECHO_ERR_INVALID_ARG;
  if (G > 16 || (d != 64 && d != 128) || (dtype != ECHO_BF16 && dtype != ECHO_F32)) return ECHO_ERR_UNSUPPORTED;
  if ((int64_t)NG * gqa_splits(k) > 0x7fffffff) return ECHO_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv) | reinterpret_cast<uintptr_t>(out)) & 15)
    return ECHO_ERR_INVALID_ARG;
  const int ns = gqa_splits(k);
  if (ns > 1 && NG > 65535) return ECHO_ERR_UNSUPPORTED;   // the merge's grid
  const size_t need = echo_sparse_gqa_workspace_bytes(NG, G, d, k);
  if (need && (!workspace || workspace_bytes < need)) return ECHO_ERR_INVALID_ARG;
  GqaPart part;
  part.o = reinterpret_cast<float *>(workspace);
  part.ml = need ? part.o + (size_t)NG * ns * G * d : nullptr;
  cudaStream_t st = (cudaStream_t)stream;
  return d == 128 ? launch_gqa<128>(q, kv, kv_rows, dtype, slot_idx, NG, G, k, scale, out, lse, part, ns, st)
                  : launch_gqa<64>(q, kv, kv_rows, dtype, slot_idx, NG, G, k, scale, out, lse, part, ns, st);
}
