// Sparse MLA decode attention over the selected cache slots (sm_103a).
//
// "ECHO: Efficient KV Cache Offloading with Lossless Prefetching ..." review page,
// "Problem and motivation": after the indexer selects the top-2048 tokens, MLA
// attention runs over their cached latent vectors (576 wide; the first 512 dims are
// the values).  Per request b and head h:
//   logit_j = scale * q[b,h,:] . c_j ;  out = softmax(logit) . c[:, :512] ;  lse.
//
// Split over the selected list: each CTA takes 256 consecutive entries of one
// request and 16 heads, streams the gathered rows through shared memory 32 at a
// time with an online softmax, and writes (o, m, l) partials; a combine kernel
// merges the splits in a fixed order.  The result depends only on the rows and
// their order in slot_idx, so attention over the cache is bitwise identical to
// attention over any buffer holding the same rows in the same order.

#include <algorithm>

#include "common.cuh"

namespace echo {

constexpr int MS_SPLIT = 256;   // selected entries per CTA
constexpr int MS_CHUNK = 32;    // rows per shared-memory chunk
constexpr int MS_HEADS = 16;    // heads per CTA
constexpr int MS_THREADS = 256;

struct MlaPart {
  float *o;   // [B, S, Hq, 512]
  float *ml;  // [B, S, Hq, 2]
};

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__global__ void __launch_bounds__(MS_THREADS)
    mla_split_kernel(const T *q, const T *kv, int kv_rows, const int32_t *slot_idx, int Hq, int k, float scale,
                     MlaPart part) {
  extern __shared__ float smf[];
  float *qs = smf;                                   // [16][576]
  float *cs = qs + MS_HEADS * KV_W;                  // [32][576]
  float *os = cs + MS_CHUNK * KV_W;                  // [16][512]
  float *lg = os + MS_HEADS * V_W;                   // [16][32]
  float *mrun = lg + MS_HEADS * MS_CHUNK;            // [16]
  float *lrun = mrun + MS_HEADS;                     // [16]
  float *corr = lrun + MS_HEADS;                     // [16]
  __shared__ int32_t slots[MS_CHUNK];

  const int s = blockIdx.x, hg = blockIdx.y, b = blockIdx.z;
  const int S = gridDim.x;
  const int h0 = hg * MS_HEADS;
  const int nh = min(MS_HEADS, Hq - h0);
  const int tid = threadIdx.x;
  const int j0 = s * MS_SPLIT, j1 = min(k, j0 + MS_SPLIT);

  for (int i = tid; i < MS_HEADS * KV_W; i += MS_THREADS) {
    const int h = i / KV_W, d = i % KV_W;
    qs[i] = h < nh ? to_f(q[((int64_t)b * Hq + h0 + h) * KV_W + d]) : 0.f;
  }
  for (int i = tid; i < MS_HEADS * V_W; i += MS_THREADS) os[i] = 0.f;
  if (tid < MS_HEADS) { mrun[tid] = -INFINITY; lrun[tid] = 0.f; }

  for (int c0 = j0; c0 < j1; c0 += MS_CHUNK) {
    __syncthreads();
    if (tid < MS_CHUNK) {
      const int j = c0 + tid;
      int32_t g = j < j1 ? slot_idx[(int64_t)b * k + j] : -1;
      if (g >= kv_rows) g = -1;
      slots[tid] = g;
    }
    __syncthreads();
    for (int i = tid; i < MS_CHUNK * KV_W; i += MS_THREADS) {
      const int r = i / KV_W, d = i % KV_W;
      const int32_t g = slots[r];
      cs[i] = g >= 0 ? to_f(kv[(int64_t)g * KV_W + d]) : 0.f;
    }
    __syncthreads();
    for (int i = tid; i < MS_HEADS * MS_CHUNK; i += MS_THREADS) {
      const int h = i / MS_CHUNK, r = i % MS_CHUNK;
      float acc = 0.f;
      const float *qh = qs + h * KV_W, *cr = cs + r * KV_W;
      for (int d = 0; d < KV_W; ++d) acc = fmaf(qh[d], cr[d], acc);
      lg[i] = (slots[r] >= 0 && h < nh) ? acc * scale : -INFINITY;
    }
    __syncthreads();
    if (tid < MS_HEADS) {
      float mx = mrun[tid];
      for (int r = 0; r < MS_CHUNK; ++r) mx = fmaxf(mx, lg[tid * MS_CHUNK + r]);
      float sum = 0.f;
      for (int r = 0; r < MS_CHUNK; ++r) {
        const float x = lg[tid * MS_CHUNK + r];
        const float p = (x == -INFINITY) ? 0.f : expf(x - mx);
        lg[tid * MS_CHUNK + r] = p;
        sum += p;
      }
      const float c = (mrun[tid] == -INFINITY) ? 0.f : expf(mrun[tid] - mx);
      corr[tid] = c;
      lrun[tid] = lrun[tid] * c + sum;
      mrun[tid] = mx;
    }
    __syncthreads();
    for (int i = tid; i < MS_HEADS * V_W; i += MS_THREADS) {
      const int h = i / V_W, d = i % V_W;
      float acc = os[i] * corr[h];
      const float *p = lg + h * MS_CHUNK;
      for (int r = 0; r < MS_CHUNK; ++r) acc = fmaf(p[r], cs[r * KV_W + d], acc);
      os[i] = acc;
    }
  }
  __syncthreads();
  for (int i = tid; i < nh * V_W; i += MS_THREADS) {
    const int h = i / V_W, d = i % V_W;
    part.o[(((int64_t)b * S + s) * Hq + h0 + h) * V_W + d] = os[i];
  }
  if (tid < nh) {
    part.ml[(((int64_t)b * S + s) * Hq + h0 + tid) * 2 + 0] = mrun[tid];
    part.ml[(((int64_t)b * S + s) * Hq + h0 + tid) * 2 + 1] = lrun[tid];
  }
}

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Merge the splits of one (request, head) in split order.
template <typename T>
__global__ void mla_combine_kernel(MlaPart part, int S, int Hq, T *out, float *lse) {
  const int h = blockIdx.x, b = blockIdx.y;
  float M = -INFINITY;
  for (int s = 0; s < S; ++s) M = fmaxf(M, part.ml[(((int64_t)b * S + s) * Hq + h) * 2]);
  float Lsum = 0.f;
  for (int s = 0; s < S; ++s) {
    const float m = part.ml[(((int64_t)b * S + s) * Hq + h) * 2];
    if (m != -INFINITY) Lsum += expf(m - M) * part.ml[(((int64_t)b * S + s) * Hq + h) * 2 + 1];
  }
  for (int d = threadIdx.x; d < V_W; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s) {
      const float m = part.ml[(((int64_t)b * S + s) * Hq + h) * 2];
      if (m != -INFINITY) acc += expf(m - M) * part.o[(((int64_t)b * S + s) * Hq + h) * V_W + d];
    }
    out[((int64_t)b * Hq + h) * V_W + d] = from_f<T>(Lsum > 0.f ? acc / Lsum : 0.f);
  }
  if (threadIdx.x == 0) lse[(int64_t)b * Hq + h] = Lsum > 0.f ? M + logf(Lsum) : -INFINITY;
}

static int mla_splits(int k) { return (k + MS_SPLIT - 1) / MS_SPLIT; }

}  // namespace echo

using namespace echo;

extern "C" size_t echo_sparse_mla_workspace_bytes(int32_t B, int32_t Hq, int32_t k) {
  if (B <= 0 || Hq <= 0 || k <= 0) return 0;
  const size_t S = (size_t)mla_splits(k);
  return (size_t)B * S * Hq * (V_W + 2) * sizeof(float);
}

extern "C" echo_status_t echo_sparse_mla_decode(const void *q, const void *kv, int32_t kv_rows, int32_t dtype,
                                                const int32_t *slot_idx, int32_t B, int32_t Hq, int32_t k,
                                                float scale, void *out, float *lse, void *workspace,
                                                size_t workspace_bytes, echo_stream_t stream) {
  if (!q || !kv || !slot_idx || !out || !lse || !workspace || B <= 0 || Hq <= 0 || k <= 0 || kv_rows <= 0)
    return ECHO_ERR_INVALID_ARG;
  if (Hq > 128) return ECHO_ERR_UNSUPPORTED;
  if (workspace_bytes < echo_sparse_mla_workspace_bytes(B, Hq, k)) return ECHO_ERR_INVALID_ARG;
  const int S = mla_splits(k);
  MlaPart part;
  part.o = reinterpret_cast<float *>(workspace);
  part.ml = part.o + (size_t)B * S * Hq * V_W;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t smem = sizeof(float) * (MS_HEADS * KV_W + MS_CHUNK * KV_W + MS_HEADS * V_W + MS_HEADS * MS_CHUNK +
                                       3 * MS_HEADS);
  dim3 grid(S, (Hq + MS_HEADS - 1) / MS_HEADS, B);
  if (dtype == ECHO_F32) {
    ECHO_CUDA_OK(cudaFuncSetAttribute(mla_split_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    mla_split_kernel<float><<<grid, MS_THREADS, smem, st>>>((const float *)q, (const float *)kv, kv_rows, slot_idx,
                                                            Hq, k, scale, part);
    ECHO_LAUNCH_OK();
    mla_combine_kernel<float><<<dim3(Hq, B), 128, 0, st>>>(part, S, Hq, (float *)out, lse);
  } else if (dtype == ECHO_BF16) {
    ECHO_CUDA_OK(cudaFuncSetAttribute(mla_split_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)smem));
    mla_split_kernel<__nv_bfloat16><<<grid, MS_THREADS, smem, st>>>(
        (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)kv, kv_rows, slot_idx, Hq, k, scale, part);
    ECHO_LAUNCH_OK();
    mla_combine_kernel<__nv_bfloat16><<<dim3(Hq, B), 128, 0, st>>>(part, S, Hq, (__nv_bfloat16 *)out, lse);
  } else {
    return ECHO_ERR_UNSUPPORTED;
  }
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}
