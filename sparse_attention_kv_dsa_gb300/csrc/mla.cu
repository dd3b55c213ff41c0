// Sparse MLA decode attention over the selected cache slots (sm_103a).
//
// "ECHO: Efficient KV Cache Offloading with Lossless Prefetching ..." review page,
// "Problem and motivation": after the indexer selects the top-2048 tokens, MLA
// attention runs over their cached latent vectors (576 wide; the first 512 dims are
// the values).  Per request b and head h:
//   logit_j = scale * q[b,h,:] . c_j ;  out = softmax(logit) . c[:, :512] ;  lse.
//
// Split over the selected list: bf16 (tensor cores) takes 512 consecutive entries of
// one request per CTA with all 128 heads; float32 (SIMT) takes 256 entries and 16
// heads per CTA, streaming the gathered rows through shared memory 32 at a time with
// an online softmax.  Both write (o, m, l) partials, and a combine kernel merges the
// splits in a fixed order.  The result depends only on the rows and their order in
// slot_idx, so attention over the cache is bitwise identical to attention over any
// buffer holding the same rows in the same order.

#include <algorithm>
#include <atomic>
#include <cudaTypedefs.h>

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

// ===================================================== bf16 tensor-core path ==
struct TcPart {
  __nv_bfloat16 *o;   // [B, S, 128, 512] normalised partial outputs
  float *ml;          // [B, S, 128, 2]
};

// 16 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// tcgen05.mma kind::f16 with A (M x 16) read from TMEM at a_tmem
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate));
}

// CTA = (request b, split s of 512 selected entries), all 128 heads, one CTA per SM
// (512 TMEM columns).  The 512 entries are two regions of 256 TMEM columns.
//   phase 1  S[128 x 512] = Q . C^T over nine 64-dim chunks x two token halves:
//            Q chunk by TMA (once per chunk), the gathered rows of one half by
//            cp.async into the 128-byte-swizzled layout; tcgen05.mma kind::f16
//            M=128 N=256 K=16 into region 0 (tokens 0-255) or 1 (256-511).
//   softmax  over all 512 entries at once: warps 0-3 read region 0, warps 4-7 region
//            1 (one head row per thread), the row max and sum are exchanged through
//            shared memory, and bf16 P goes back into TMEM over logits already read
//            (token t of region r to column 256 r + (t mod 256) / 2, so P fills the first
//            128 columns of each region).
//   phase 2  O = P . V in four 128-dim blocks, each over four 128-token quarters; A = P
//            from TMEM, B = 16-token x 128-dim pieces (MN-major, two 64-dim atoms) of a
//            stage; two O buffers (columns 128-255 and 384-511) so the epilogue of block
//            j overlaps the MMAs of block j+1.  The epilogue writes O / l as bf16
//            partials plus (m, l) per head, in the layout the combine reads.
// Every load stage is 32 KB in 128-byte rows (row r at 128 r, its 16-byte chunk c at
// (c ^ (r & 7)) * 16): a K stage of phase 1 is 256 rows x 64 dims, a V stage of phase 2
// is two atoms of 128 rows x 64 dims (the block's two dim halves, 16 KB apart); both go
// through one ring of five slots (160 KB in flight), and the V rows start loading as
// soon as phase 1 frees slots.
// Roles: warps 0-3 softmax of region 0 and the epilogues, warps 4-7 softmax of
// region 1, warp 8 issues the MMAs from lane 0 and the Q chunks' TMA from lane 1
// (three chunks ahead, apart from the row loads), warps 9-16 only load rows.  Each
// loader thread ends a stage with cp.async.mbarrier.arrive.noinc on the slot's
// barrier (256 arrivals), which fires once its copies have landed: the loaders never
// wait for their own copies; the MMA thread fences them for the tensor cores.
constexpr int T2_T = 512;                     // selected entries per CTA
constexpr int T2_LOADERS = 256;               // loader threads (warps 9-16)
constexpr int T2_THREADS = 9 * 32 + T2_LOADERS;
constexpr int T2_QST = 3, T2_SLOTS = 5;
constexpr int T2_QCH = 128 * 128;             // Q chunk bytes
constexpr int T2_SCH = 256 * 128;             // stage: 256 rows x 64 dims
constexpr int T2_NK = 18;                     // phase-1 stages: 9 chunks x 2 halves
constexpr int T2_NS = T2_NK + 16;             // + phase-2 stages: 4 blocks x 4 quarters
constexpr int T2_SOFF = T2_QST * T2_QCH;
constexpr int T2_REGION = T2_SOFF + T2_SLOTS * T2_SCH;     // 192 KB

struct T2Shared {
  uint64_t qfull[T2_QST], qempty[T2_QST], full[T2_SLOTS], empty[T2_SLOTS];
  uint64_t s_full, p_full, o_full[2], o_empty[2];
  uint32_t tmem_base;
  int fail;
  int32_t slots[T2_T];
  uint32_t vmask[T2_T / 32];
  float mpart[2][128], lpart[2][128];
};
constexpr size_t T2_SMEM = 1024 + T2_REGION + sizeof(T2Shared);
static_assert(T2_SMEM <= 227 * 1024, "one CTA per SM");

__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// TMEM column of the bf16 pair holding tokens t, t+1 (t even) of the 512 entries
__device__ __forceinline__ uint32_t p2_col(int t) {
  return (uint32_t)(256 * (t >> 8) + ((t & 255) >> 1));
}

__global__ void __launch_bounds__(T2_THREADS, 1)
    mla_tc2_kernel(const __grid_constant__ CUtensorMap qmap, const __nv_bfloat16 *kv, int kv_rows,
                   const int32_t *slot_idx, int k, float scale, TcPart part) {
  extern __shared__ unsigned char t2_raw[];
  unsigned char *R = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(t2_raw) + 1023) & ~uintptr_t(1023));
  T2Shared &S = *reinterpret_cast<T2Shared *>(R + T2_REGION);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s = blockIdx.x, b = blockIdx.y, nsplit = gridDim.x;
  const int j0 = s * T2_T;

  if (tid == 0) {
    for (int i = 0; i < T2_QST; ++i) { mbar_init(&S.qfull[i], 1); mbar_init(&S.qempty[i], 1); }
    for (int i = 0; i < T2_SLOTS; ++i) { mbar_init(&S.full[i], T2_LOADERS); mbar_init(&S.empty[i], 1); }
    mbar_init(&S.s_full, 1);
    mbar_init(&S.p_full, 256);
    for (int i = 0; i < 2; ++i) { mbar_init(&S.o_full[i], 1); mbar_init(&S.o_empty[i], 128); }
    S.fail = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < T2_T; i += T2_THREADS) {
    const int j = j0 + i;
    int32_t g = j < k ? slot_idx[(int64_t)b * k + j] : -1;
    g = (g >= 0 && g < kv_rows) ? g : -1;
    S.slots[i] = g;
  }
  __syncthreads();
  for (int w = warp; w < T2_T / 32; w += T2_THREADS / 32) {   // 16 mask words over 13 warps
    const uint32_t bal = __ballot_sync(0xffffffffu, S.slots[w * 32 + lane] >= 0);
    if (lane == 0) S.vmask[w] = bal;
  }
  if (warp == 8) {
    tmem_alloc(&S.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  bool ok = true;

  if (warp >= 9) {
    // ------------------------------------------------------------ loads --
    // thread lt copies chunk c = lt & 7 of rows (lt >> 3) + 32 i of each stage: the
    // same rows in every stage of a half, so their slots are read once into registers
    constexpr int RPT = 256 * 8 / T2_LOADERS;          // rows per thread and stage (8)
    const int lt = tid - 9 * 32, c = lt & 7, r0 = lt >> 3;
    int32_t rows[2][RPT];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < RPT; ++i) rows[h][i] = S.slots[h * 256 + r0 + 32 * i];
    for (int g = 0; g < T2_NS && ok; ++g) {
      const int sl = g % T2_SLOTS;
      if (!mbar_wait(&S.empty[sl], ((g / T2_SLOTS) & 1) ^ 1)) { ok = false; break; }
      unsigned char *sb = R + T2_SOFF + sl * T2_SCH;
      if (g < T2_NK) {
        const int dc = g >> 1, half = g & 1;           // dims 64 dc .., tokens 256 half ..
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const int r = r0 + 32 * i;
          const int32_t row = half ? rows[1][i] : rows[0][i];
          const __nv_bfloat16 *src = kv + (int64_t)(row >= 0 ? row : 0) * KV_W + dc * 64 + c * 8;
          cp_async_16(sb + r * 128 + ((c ^ (r & 7)) << 4), src, row >= 0 ? 16u : 0u);
        }
      } else {
        // value stage: tokens 128 q .. of dims 128 j .., two 64-dim atoms of 128 rows
        const int gv = g - T2_NK, j = gv >> 2, q = gv & 3;
        const int cc = lt & 15, atom = cc >> 3, c2 = cc & 7, rr0 = lt >> 4;
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const int r = rr0 + 16 * i;
          const int32_t row = S.slots[128 * q + r];
          const __nv_bfloat16 *src = kv + (int64_t)(row >= 0 ? row : 0) * KV_W + j * 128 + atom * 64 + c2 * 8;
          cp_async_16(sb + atom * (128 * 128) + r * 128 + ((c2 ^ (r & 7)) << 4), src, row >= 0 ? 16u : 0u);
        }
      }
      cp_async_arrive(&S.full[sl]);
    }
    cp_async_wait_all();                               // nothing of ours stays in flight at the end
  } else if (warp == 8) {
    if (lane == 1) {
      // ------------------------------------------------- Q chunks (TMA) --
      int issued = 0;
      for (int dc = 0; dc < 9; ++dc) {
        const int qs = dc % T2_QST;
        if (!mbar_wait(&S.qempty[qs], ((dc / T2_QST) & 1) ^ 1)) { ok = false; break; }
        mbar_arrive_expect_tx(&S.qfull[qs], T2_QCH);
        tma_load_2d(R + qs * T2_QCH, &qmap, &S.qfull[qs], dc * 64, b * 128);
        issued = dc + 1;
      }
      // on a failure, the chunks in flight land before the CTA ends (bounded waits)
      for (int dc = ok ? issued : max(0, issued - T2_QST); !ok && dc < issued; ++dc)
        mbar_wait(&S.qfull[dc % T2_QST], (dc / T2_QST) & 1);
    }
    if (lane == 0) {
      // --------------------------------------------------------------- MMA --
      constexpr uint32_t id1 = instr_desc(FMT_BF16, FMT_BF16, 0, 0, 128, 256);
      constexpr uint32_t id2 = instr_desc(FMT_BF16, FMT_BF16, 0, 1, 128, 128);
      for (int g = 0; g < T2_NS && ok; ++g) {
        const int sl = g % T2_SLOTS;
        const uint32_t sa = smem_u32(R + T2_SOFF + sl * T2_SCH);
        if (g < T2_NK) {
          // S[:, half] += Q chunk dc . rows^T
          const int dc = g >> 1, half = g & 1, qs = dc % T2_QST;
          if (!mbar_wait(&S.qfull[qs], (dc / T2_QST) & 1) || !mbar_wait(&S.full[sl], (g / T2_SLOTS) & 1)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();                    // the loaders' cp.async writes, for the tensor cores
          tc_fence_after();
          const uint64_t ad = smem_desc(smem_u32(R + qs * T2_QCH), 16, 1024, LAYOUT_SW128);
          const uint64_t bd = smem_desc(sa, 16, 1024, LAYOUT_SW128);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(tmem + 256 * half, ad + 2 * kk, bd + 2 * kk, id1, (dc | kk) ? 1u : 0u);
          mma_commit(&S.empty[sl]);
          if (half == 1) mma_commit(&S.qempty[qs]);
          if (g == T2_NK - 1) {
            mma_commit(&S.s_full);
            if (!mbar_wait(&S.p_full, 0)) { ok = false; break; }   // P written by the softmax
            tc_fence_after();
          }
        } else {
          // O_j += P[:, tokens of quarter q] . V[those tokens, dims of block j]
          const int gv = g - T2_NK, j = gv >> 2, q = gv & 3, ob = j & 1;
          if (q == 0 && j >= 2) {                      // this buffer's previous block is written out
            if (!mbar_wait(&S.o_empty[ob], ((j >> 1) - 1) & 1)) { ok = false; break; }
            tc_fence_after();
          }
          if (!mbar_wait(&S.full[sl], (g / T2_SLOTS) & 1)) { ok = false; break; }
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t d = tmem + 128u + 256u * (uint32_t)ob;
#pragma unroll
          for (int u = 0; u < 8; ++u) {                // 8 K-steps of 16 tokens; N = 128 dims in two atoms
            const int t0 = 128 * q + 16 * u;
            const uint64_t bd = smem_desc(sa + (uint32_t)(u * 16 * 128), 128 * 128, 1024, LAYOUT_SW128);
            mma_f16_ts(d, tmem + p2_col(t0), bd, id2, (q | u) ? 1u : 0u);
          }
          mma_commit(&S.empty[sl]);
          if (q == 3) mma_commit(&S.o_full[ob]);
        }
      }
    }
  } else {
    // ------------------------------------------------------- softmax --
    const int half = warp >> 2;                        // region of the 512 entries
    const int hr = (warp & 3) * 32 + lane;             // head row = TMEM lane
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t tr = trow + 256u * (uint32_t)half;
    if (!mbar_wait(&S.s_full, 0)) ok = false;
    tc_fence_after();
    float m = -INFINITY;
    for (int c0 = 0; c0 < 256; c0 += 64) {
      uint32_t r[32], r2[32];
      tmem_ld32(tr + c0, r);
      tmem_ld32(tr + c0 + 32, r2);
      tmem_wait_ld();
      const uint32_t vm = S.vmask[(half * 256 + c0) >> 5], vm2 = S.vmask[((half * 256 + c0) >> 5) + 1];
#pragma unroll
      for (int q = 0; q < 32; ++q) {
        if ((vm >> q) & 1u) m = fmaxf(m, __uint_as_float(r[q]));
        if ((vm2 >> q) & 1u) m = fmaxf(m, __uint_as_float(r2[q]));
      }
    }
    S.mpart[half][hr] = m;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    m = fmaxf(S.mpart[0][hr], S.mpart[1][hr]);
    const float c2 = scale * 1.4426950408889634f;     // scale * log2(e)
    const float mc = m * c2;
    float l = 0.f;
    auto write_p = [&](int c0, const uint32_t (&r)[32], uint32_t vm) {
      uint32_t pk[16];
#pragma unroll
      for (int q = 0; q < 32; q += 2) {
        const float p0 = ((vm >> q) & 1u) ? exp2f(fmaf(__uint_as_float(r[q]), c2, -mc)) : 0.f;
        const float p1 = ((vm >> (q + 1)) & 1u) ? exp2f(fmaf(__uint_as_float(r[q + 1]), c2, -mc)) : 0.f;
        l += p0 + p1;
        __nv_bfloat162 v2 = __floats2bfloat162_rn(p0, p1);
        pk[q >> 1] = *reinterpret_cast<uint32_t *>(&v2);
      }
      tmem_st16(trow + p2_col(half * 256 + c0), pk);
    };
    for (int c0 = 0; c0 < 256; c0 += 64) {
      uint32_t r[32], r2[32];
      tmem_ld32(tr + c0, r);
      tmem_ld32(tr + c0 + 32, r2);
      tmem_wait_ld();
      write_p(c0, r, S.vmask[(half * 256 + c0) >> 5]);
      write_p(c0 + 32, r2, S.vmask[((half * 256 + c0) >> 5) + 1]);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&S.p_full);
    S.lpart[half][hr] = l;
    asm volatile("bar.sync 2, 256;" ::: "memory");
    l = S.lpart[0][hr] + S.lpart[1][hr];
    if (half == 0) {
      // ----------------------------------------------------- epilogues --
      // O / l of block j from its TMEM buffer to bf16 partials, stored in groups of 8
      // dims with heads innermost ([b][s][dim/8][head][8]): the 32 heads of a warp
      // write one contiguous 512-byte run per store
      const float inv = l > 0.f ? 1.f / l : 0.f;
      for (int j = 0; j < 4; ++j) {
        const int ob = j & 1;
        if (!mbar_wait(&S.o_full[ob], (j >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        __nv_bfloat16 *dst = part.o + (((int64_t)b * nsplit + s) * 64 + j * 16) * 128 * 8 + (int64_t)hr * 8;
        const uint32_t oc = trow + 128u + 256u * (uint32_t)ob;
        auto store_o = [&](int c0, const uint32_t (&v)[32]) {
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 32; q += 2) {
            __nv_bfloat162 v2 =
                __floats2bfloat162_rn(__uint_as_float(v[q]) * inv, __uint_as_float(v[q + 1]) * inv);
            pk[q >> 1] = *reinterpret_cast<uint32_t *>(&v2);
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4 *>(dst + (int64_t)((c0 >> 3) + q) * 128 * 8) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        };
        for (int hc = 0; hc < 2; ++hc) {               // the block's 128 columns in two halves
          uint32_t r[32], r2[32];
          tmem_ld32(oc + 64u * hc, r);
          tmem_ld32(oc + 64u * hc + 32, r2);
          tmem_wait_ld();
          if (hc == 1) {
            tc_fence_before();
            mbar_arrive(&S.o_empty[ob]);               // the values are in registers
          }
          store_o(64 * hc, r);
          store_o(64 * hc + 32, r2);
        }
      }
      part.ml[(((int64_t)b * nsplit + s) * 128 + hr) * 2 + 0] = m == -INFINITY ? -INFINITY : m * scale;
      part.ml[(((int64_t)b * nsplit + s) * 128 + hr) * 2 + 1] = l;
    }
  }
  if (!ok) S.fail = 1;                                // a bounded wait gave up
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8) tmem_dealloc(tmem, 512);
  if (S.fail && tid < 128) {
    // this split's partial is not valid: the combine skips a split whose max is -inf
    part.ml[(((int64_t)b * nsplit + s) * 128 + tid) * 2 + 0] = -INFINITY;
    part.ml[(((int64_t)b * nsplit + s) * 128 + tid) * 2 + 1] = 0.f;
  }
}

// Merge the bf16 partials of one (request, head) in split order.  A block of 256
// threads covers 4 heads; each thread produces 8 consecutive output dims.
template <int NSMAX>
__global__ void __launch_bounds__(256) mla_tc_combine_kernel(TcPart part, int nsplit, __nv_bfloat16 *out,
                                                             float *lse, int drop) {
  // block: two groups of 8 dims (j) x 128 heads; warp w: heads 32 (w & 3) + lane of group
  // j = 2 blockIdx.x + (w >> 2), so every load of a partial is a contiguous 512-byte run
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = 32 * (warp & 3) + lane;
  const int j = 2 * blockIdx.x + (warp >> 2);
  const float *ml = part.ml + ((int64_t)b * nsplit * 128 + h) * 2;                  // split s at ml[s * 256]
  const __nv_bfloat16 *po = part.o + (((int64_t)b * nsplit * 64 + j) * 128 + h) * 8;  // split s at po[s * 65536]
  float M = -INFINITY;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float Lsum = 0.f;
  auto add = [&](float m, float l, const uint4 &v) {
    const float w = (m == -INFINITY || l <= 0.f) ? 0.f : expf(m - M) * l;
    Lsum += w;
    const __nv_bfloat162 *p2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[2 * q] = fmaf(w, __bfloat162float(p2[q].x), acc[2 * q]);
      acc[2 * q + 1] = fmaf(w, __bfloat162float(p2[q].y), acc[2 * q + 1]);
    }
  };
  if (nsplit <= NSMAX) {
    // every split's (m, l) and partial issued together, then merged in split order
    float m[NSMAX], l[NSMAX];
    uint4 v[NSMAX];
#pragma unroll
    for (int s = 0; s < NSMAX; ++s) {
      if (s < nsplit) {
        m[s] = __ldg(ml + (int64_t)s * 256);
        l[s] = __ldg(ml + (int64_t)s * 256 + 1);
        v[s] = __ldg(reinterpret_cast<const uint4 *>(po + (int64_t)s * 64 * 128 * 8));
      }
    }
#pragma unroll
    for (int s = 0; s < NSMAX; ++s)
      if (s < nsplit) M = fmaxf(M, m[s]);
#pragma unroll
    for (int s = 0; s < NSMAX; ++s)
      if (s < nsplit) add(m[s], l[s], v[s]);
  } else {
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldg(ml + (int64_t)s * 256));
    for (int s = 0; s < nsplit; ++s)
      add(__ldg(ml + (int64_t)s * 256), __ldg(ml + (int64_t)s * 256 + 1),
          __ldg(reinterpret_cast<const uint4 *>(po + (int64_t)s * 64 * 128 * 8)));
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  uint4 o;
  __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
  for (int q = 0; q < 4; ++q) o2[q] = __floats2bfloat162_rn(acc[2 * q] * inv, acc[2 * q + 1] * inv);
  *reinterpret_cast<uint4 *>(out + ((int64_t)b * 128 + h) * V_W + 8 * j) = o;
  // the per-split logits are scaled, so M and lse are in logit units
  if (j == 0) lse[(int64_t)b * 128 + h] = Lsum > 0.f ? M + logf(Lsum) : -INFINITY;
  if (drop) {
    // The partials are dead once merged: their L2 lines are dropped without being
    // written back, so the next kernels' streams do not pay for evicting them.  Each
    // split's chunks of this warp are 512 contiguous bytes (4 lines), read only here;
    // lane i drops line i & 3 of splits (i >> 2), (i >> 2) + 8, ...
    __syncwarp();
    const __nv_bfloat16 *p0 = po - lane * 8;
    for (int s = lane >> 2; s < nsplit; s += 8) {
      const __nv_bfloat16 *line = p0 + (int64_t)s * 64 * 128 * 8 + (lane & 3) * 64;
      asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
    }
  }
}

// Q as a 2-D bf16 tensor [rows, 576] with a [128 rows x 64 dims] box, 128-byte swizzle.
static bool make_q_map(CUtensorMap *m, const void *base, uint64_t rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 enc = nullptr;
  if (!enc) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return false;
    enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  const cuuint64_t dims[2] = {KV_W, rows};
  const cuuint64_t strides[1] = {KV_W * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

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
    if (Hq != 128) return ECHO_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15) return ECHO_ERR_INVALID_ARG;
    const int ns = (k + T2_T - 1) / T2_T;
    if (ns > 64) return ECHO_ERR_UNSUPPORTED;
    TcPart tp;
    tp.o = reinterpret_cast<__nv_bfloat16 *>(workspace);
    tp.ml = reinterpret_cast<float *>(tp.o + (size_t)B * ns * 128 * 512);
    CUtensorMap qmap;
    if (!make_q_map(&qmap, q, (uint64_t)B * 128)) return ECHO_ERR_CUDA;
    ECHO_CUDA_OK(cudaFuncSetAttribute(mla_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)T2_SMEM));
    mla_tc2_kernel<<<dim3(ns, B), T2_THREADS, T2_SMEM, st>>>(qmap, (const __nv_bfloat16 *)kv, kv_rows, slot_idx, k,
                                                             scale, tp);
    ECHO_LAUNCH_OK();
    // the partials' lines are dropped after the merge when they are whole lines
    const int drop = (reinterpret_cast<uintptr_t>(workspace) & 127) == 0;
    mla_tc_combine_kernel<8><<<dim3(32, B), 256, 0, st>>>(tp, ns, (__nv_bfloat16 *)out, lse, drop);
  } else {
    return ECHO_ERR_UNSUPPORTED;
  }
  ECHO_LAUNCH_OK();
  return ECHO_OK;
}

// ----------------------------------------------- variant without allocation --
// For callers that may not allocate device memory: the split partials go to a
// scratch array compiled into the library instead of a caller workspace.  Every
// GPU that loads the library holds the array until the process exits.
namespace {
static __device__ __align__(256) unsigned char g_mla_noalloc_scratch[ECHO_MLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
// device address of the array, per device; host threads that make their first call
// on a device at the same time may both look it up, and both store the same value
std::atomic<void *> g_scratch_addr[kMaxDevices];
}  // namespace

extern "C" echo_status_t echo_sparse_mla_decode_noalloc(const void *q, const void *kv, int32_t kv_rows,
                                                        int32_t dtype, const int32_t *slot_idx, int32_t B,
                                                        int32_t Hq, int32_t k, float scale, void *out, float *lse,
                                                        echo_stream_t stream) {
  if (!q || !kv || !slot_idx || !out || !lse || B <= 0 || Hq <= 0 || k <= 0 || kv_rows <= 0)
    return ECHO_ERR_INVALID_ARG;
  const size_t need = echo_sparse_mla_workspace_bytes(B, Hq, k);
  if (need == 0) return ECHO_ERR_INVALID_ARG;
  if (need > (size_t)ECHO_MLA_NOALLOC_SCRATCH_BYTES) return ECHO_ERR_SCRATCH_LIMIT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ECHO_ERR_CUDA;
  void *scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!scratch) {
    // host code cannot use the array's name as a device address: look it up once
    // per device, with that device current
    if (cudaGetSymbolAddress(&scratch, g_mla_noalloc_scratch) != cudaSuccess || !scratch) return ECHO_ERR_CUDA;
    g_scratch_addr[dev].store(scratch, std::memory_order_release);
  }
  return echo_sparse_mla_decode(q, kv, kv_rows, dtype, slot_idx, B, Hq, k, scale, out, lse, scratch,
                                (size_t)ECHO_MLA_NOALLOC_SCRATCH_BYTES, stream);
}
