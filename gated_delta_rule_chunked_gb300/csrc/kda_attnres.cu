// kda_attnres.cu -- Attention Residuals: softmax-weighted sum of up to 9 sources per token,
// scored by a pseudo-query against each RMS-normalised source, forward and backward.
//
//   r_i = (mean_c x_ic^2 + eps)^(-1/2),  logit_i = r_i (w . x_i),  alpha = softmax(logit),
//   out = sum_i alpha_i x_i.
// Backward with g = d_out, n_i = r_i x_i (so logit_i = w . n_i):
//   da_i = g . x_i,  dlogit_i = alpha_i (da_i - sum_j alpha_j da_j),
//   dx_i = alpha_i g + r_i dlogit_i (w - x_i r_i logit_i / d)     (RMS-norm backward: the
//          projection of dn_i = dlogit_i w onto n_i is dlogit_i logit_i / d per element),
//   dw   = sum_tokens sum_i dlogit_i r_i x_i.
// Memory-bound. Forward: a cluster of 4 CTAs per token, each holding a quarter of the
// channels of every source in registers, so the sources are read from memory once; the
// 2S per-token sums meet through distributed shared memory (each CTA adds the four partial
// sums in rank order, so all four see the same statistics), and each CTA writes its quarter
// of the output. Nothing else is materialised beyond three [T, S] fp32 statistics.
// Backward: each token's sources are read twice by the same CTA (the second pass is
// served from L1/L2). dw is reduced deterministically: fixed per-CTA partials over a
// fixed token assignment, then a fixed-order sum.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int AR_MAXS = 9;
constexpr int AR_CPT = 4;        // 16-byte chunks per thread and source
constexpr int AR_MAXW = 32;      // warps per CTA at most

namespace {
template <typename IO> struct Vec;
template <> struct Vec<bf16> {
  static constexpr int N = 8;   // elements per 16-byte chunk
  static __device__ __forceinline__ void load(const void *p, float (&x)[8]) { unpack(*reinterpret_cast<const uint4 *>(p), x); }
  static __device__ __forceinline__ void unpack(const uint4 u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
      x[2 * e] = f.x;
      x[2 * e + 1] = f.y;
    }
  }
  static __device__ __forceinline__ void store(void *p, const float (&x)[8]) {
    uint4 u;
    uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
      w[e] = *reinterpret_cast<const uint32_t *>(&b);
    }
    *reinterpret_cast<uint4 *>(p) = u;
  }
};
template <> struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const void *p, float (&x)[4]) { unpack(*reinterpret_cast<const uint4 *>(p), x); }
  static __device__ __forceinline__ void unpack(const uint4 u, float (&x)[4]) {
    x[0] = __uint_as_float(u.x); x[1] = __uint_as_float(u.y); x[2] = __uint_as_float(u.z); x[3] = __uint_as_float(u.w);
  }
  static __device__ __forceinline__ void store(void *p, const float (&x)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
  }
};

// Threads per CTA: about AR_CPT chunks each, in whole warps.
__host__ __device__ inline int ar_threads(int nch) {
  int t = (nch + AR_CPT - 1) / AR_CPT;
  t = (t + 31) / 32 * 32;
  return t < 32 ? 32 : (t > 1024 ? 1024 : t);
}

// Sum `n` per-thread values over the CTA (fixed order); results in out[0..n) for every thread.
template <int NMAX>
__device__ __forceinline__ void block_sum(float (&v)[NMAX], int n, float *red, float *out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int i = 0; i < NMAX; ++i)
    if (i < n) {
      float x = v[i];
#pragma unroll
      for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      if (lane == 0) red[warp * NMAX + i] = x;
    }
  __syncthreads();
  if ((int)threadIdx.x < n) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += red[w * NMAX + threadIdx.x];
    out[threadIdx.x] = s;
  }
  __syncthreads();
}
}  // namespace

// Cluster helpers: this CTA's rank, a peer's copy of a shared variable, the split barrier.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ float ld_peer(const float *p, uint32_t rank) {
  uint32_t a;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory"); }

constexpr int AR_CL = 4;   // CTAs per token

// CTA (token t, quarter q) owns channel chunks [q per, (q+1) per): one thread copies the S
// source slices into shared memory with bulk copies (per x 16 bytes each), then the CTA's
// threads walk the chunks, twice (sums, then the output), from shared memory.
template <typename IO>
__global__ void __cluster_dims__(AR_CL, 1, 1) __launch_bounds__(256) attnres_fwd_kernel(AttnresParams p) {
  constexpr int N = Vec<IO>::N;
  extern __shared__ __align__(128) char ar_smem[];
  __shared__ float red[8 * 2 * AR_MAXS], part[2 * AR_MAXS], al[AR_MAXS];
  __shared__ __align__(8) uint64_t bar;
  const long long t = blockIdx.x / AR_CL;
  const uint32_t q = cluster_rank();
  const int S = p.S, d = p.dim, nch = d / N, per = (nch + AR_CL - 1) / AR_CL;
  const int cbeg = (int)q * per, cend = min(cbeg + per, nch), nown = max(cend - cbeg, 0);
  uint4 *xs = reinterpret_cast<uint4 *>(ar_smem);   // [S][per] 16-byte chunks
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_expect_tx(&bar, (uint32_t)(S * nown * 16));
    if (nown > 0)
      for (int i = 0; i < S; ++i)
        bulk_g2s(xs + (size_t)i * per, static_cast<const IO *>(p.src[i]) + t * d + (size_t)cbeg * N, (uint32_t)(nown * 16),
                 &bar);
  }
  float acc[2 * AR_MAXS];
#pragma unroll
  for (int i = 0; i < 2 * AR_MAXS; ++i) acc[i] = 0.f;
  const bool ok = mbar_wait(&bar, 0);
  if (!ok && threadIdx.x == 0) report(p.status, ERR_TIMEOUT);   // carry on: the cluster barriers below must be met
  for (int c = threadIdx.x; c < nown; c += blockDim.x) {
    float w[N], x[N];
#pragma unroll
    for (int e = 0; e < N; ++e) w[e] = p.w[(cbeg + c) * N + e];
#pragma unroll
    for (int i = 0; i < AR_MAXS; ++i)
      if (i < S) {
        Vec<IO>::unpack(xs[(size_t)i * per + c], x);
#pragma unroll
        for (int e = 0; e < N; ++e) {
          acc[2 * i] = fmaf(x[e], x[e], acc[2 * i]);
          acc[2 * i + 1] = fmaf(w[e], x[e], acc[2 * i + 1]);
        }
      }
  }
  block_sum(acc, 2 * S, red, part);   // this quarter's sums, visible to the cluster after the barrier
  cluster_arrive();
  cluster_wait();
  if (threadIdx.x < 32) {   // warp 0: lane k gathers sum k over the cluster (rank order: identical in every CTA)
    const int k = threadIdx.x;
    float v = 0.f;
    if (k < 2 * S)
#pragma unroll
      for (uint32_t r = 0; r < AR_CL; ++r) v += ld_peer(&part[k], r);
    const float sq = __shfl_sync(0xffffffffu, v, (2 * k) & 31), wx = __shfl_sync(0xffffffffu, v, (2 * k + 1) & 31);
    const bool src = k < S;
    const float r = rsqrtf(sq / d + p.eps), lg = src ? r * wx : -INFINITY;   // lane i: source i
    float mx = lg;
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float ex = src ? __expf(lg - mx) : 0.f;
    float z = ex;
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (src) {
      al[k] = ex / z;
      if (q == 0) {
        p.rstd[t * S + k] = r;
        p.logit[t * S + k] = lg;
        p.alpha[t * S + k] = ex / z;
      }
    }
  }
  cluster_arrive();   // done reading the peers' sums; the matching wait comes before exit
  __syncthreads();
  for (int c = threadIdx.x; c < nown; c += blockDim.x) {
    float o[N], x[N];
#pragma unroll
    for (int e = 0; e < N; ++e) o[e] = 0.f;
#pragma unroll
    for (int i = 0; i < AR_MAXS; ++i)
      if (i < S) {
        Vec<IO>::unpack(xs[(size_t)i * per + c], x);
#pragma unroll
        for (int e = 0; e < N; ++e) o[e] = fmaf(al[i], x[e], o[e]);
      }
    Vec<IO>::store(static_cast<IO *>(p.out) + t * d + (size_t)(cbeg + c) * N, o);
  }
  cluster_wait();   // no CTA leaves while a peer may still read its sums
}

// Persistent: CTA b takes tokens b, b + grid, ...; each thread owns fixed channel chunks
// (c = tid + blockDim j, j < MAXJ) and keeps their dw partial sums; partial[b][c] at the end.
template <typename IO, int MAXJ>
__global__ void __launch_bounds__(1024) attnres_bwd_kernel(AttnresParams p) {
  constexpr int N = Vec<IO>::N;
  __shared__ float red[AR_MAXW * AR_MAXS], tot[AR_MAXS];
  const int S = p.S, d = p.dim, nch = d / N;
  const float inv_d = 1.f / d;
  float dw[MAXJ][N];
#pragma unroll
  for (int j = 0; j < MAXJ; ++j)
#pragma unroll
    for (int e = 0; e < N; ++e) dw[j][e] = 0.f;
  for (long long t = blockIdx.x; t < p.T; t += gridDim.x) {
    float al[AR_MAXS], rs[AR_MAXS], lg[AR_MAXS], da[AR_MAXS];
#pragma unroll
    for (int i = 0; i < AR_MAXS; ++i) {
      al[i] = i < S ? p.alpha[t * S + i] : 0.f;
      rs[i] = i < S ? p.rstd[t * S + i] : 0.f;
      lg[i] = i < S ? p.logit[t * S + i] : 0.f;
      da[i] = 0.f;
    }
    // pass 1: da_i = g . x_i
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      const int c = threadIdx.x + blockDim.x * j;
      if (c < nch) {
        float g[N], x[N];
        Vec<IO>::load(static_cast<const IO *>(p.dout) + t * d + c * N, g);
#pragma unroll
        for (int i = 0; i < AR_MAXS; ++i)
          if (i < S) {
            Vec<IO>::load(static_cast<const IO *>(p.src[i]) + t * d + c * N, x);
#pragma unroll
            for (int e = 0; e < N; ++e) da[i] = fmaf(g[e], x[e], da[i]);
          }
      }
    }
    block_sum(da, S, red, tot);
    float mean = 0.f, dl[AR_MAXS];
#pragma unroll
    for (int i = 0; i < AR_MAXS; ++i)
      if (i < S) mean = fmaf(al[i], tot[i], mean);
#pragma unroll
    for (int i = 0; i < AR_MAXS; ++i) dl[i] = i < S ? al[i] * (tot[i] - mean) : 0.f;
    // pass 2: dx_i and the dw partials
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      const int c = threadIdx.x + blockDim.x * j;
      if (c < nch) {
        float g[N], w[N], x[N], dx[N];
        Vec<IO>::load(static_cast<const IO *>(p.dout) + t * d + c * N, g);
#pragma unroll
        for (int e = 0; e < N; ++e) w[e] = p.w[c * N + e];
#pragma unroll
        for (int i = 0; i < AR_MAXS; ++i)
          if (i < S) {
            Vec<IO>::load(static_cast<const IO *>(p.src[i]) + t * d + c * N, x);
            const float a = rs[i] * dl[i], b = rs[i] * lg[i] * inv_d;
#pragma unroll
            for (int e = 0; e < N; ++e) {
              dx[e] = fmaf(al[i], g[e], a * (w[e] - x[e] * b));
              dw[j][e] = fmaf(a, x[e], dw[j][e]);
            }
            Vec<IO>::store(static_cast<IO *>(p.dsrc[i]) + t * d + c * N, dx);
          }
      }
    }
    __syncthreads();   // `tot` is reused by the next token
  }
#pragma unroll
  for (int j = 0; j < MAXJ; ++j) {
    const int c = threadIdx.x + blockDim.x * j;
    if (c < nch)
#pragma unroll
      for (int e = 0; e < N; ++e) p.partial[(size_t)blockIdx.x * d + c * N + e] = dw[j][e];
  }
}

__global__ void attnres_dw_reduce_kernel(const float *partial, int nparts, int d, float *dw) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  float s = 0.f;
  for (int b = 0; b < nparts; ++b) s += partial[(size_t)b * d + c];
  dw[c] = s;
}

// Backward grid: as many CTAs as fit on the device at once (the dw partials are per CTA).
int attnres_bwd_ctas(long long T, bool f32, int dim) {
  int dev = 0, sms = 0, per = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 1;
  const int threads = ar_threads(dim / (f32 ? 4 : 8));
  const cudaError_t e = f32 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, attnres_bwd_kernel<float, AR_CPT>, threads, 0)
                            : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, attnres_bwd_kernel<bf16, AR_CPT>, threads, 0);
  if (e != cudaSuccess || per < 1) per = 1;
  const long long cap = (long long)sms * per;
  return (int)(T < cap ? (T > 0 ? T : 1) : cap);
}

cudaError_t launch_attnres_fwd(const AttnresParams &p, bool f32, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  const int per = (p.dim / (f32 ? 4 : 8) + AR_CL - 1) / AR_CL;   // chunks per CTA
  const int smem = p.S * per * 16;
  int threads = (per + 31) / 32 * 32;
  threads = threads < 32 ? 32 : (threads > 256 ? 256 : threads);
  const unsigned grid = (unsigned)(p.T * AR_CL);
  auto kern = f32 ? attnres_fwd_kernel<float> : attnres_fwd_kernel<bf16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, threads, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attnres_bwd(const AttnresParams &p, bool f32, cudaStream_t s) {
  const int nparts = attnres_bwd_ctas(p.T, f32, p.dim);
  if (p.T > 0) {
    const int threads = ar_threads(p.dim / (f32 ? 4 : 8));   // at most AR_CPT chunks per thread
    if (f32)
      attnres_bwd_kernel<float, AR_CPT><<<nparts, threads, 0, s>>>(p);
    else
      attnres_bwd_kernel<bf16, AR_CPT><<<nparts, threads, 0, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = cudaMemsetAsync(p.partial, 0, (size_t)p.dim * sizeof(float), s);
    if (e != cudaSuccess) return e;
  }
  attnres_dw_reduce_kernel<<<(p.dim + 255) / 256, 256, 0, s>>>(p.partial, nparts, p.dim, p.dw);
  return cudaGetLastError();
}

}  // namespace kda
