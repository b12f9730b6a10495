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
// Memory-bound: each token's sources are read twice by the same CTA (the second pass is
// served from L1/L2), the output written once, nothing else materialised beyond three
// [T, S] fp32 statistics. dw is reduced deterministically: fixed per-CTA partials over a
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
  static __device__ __forceinline__ void load(const void *p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
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
  static __device__ __forceinline__ void load(const void *p, float (&x)[4]) {
    const float4 f = *reinterpret_cast<const float4 *>(p);
    x[0] = f.x; x[1] = f.y; x[2] = f.z; x[3] = f.w;
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

template <typename IO>
__global__ void __launch_bounds__(1024) attnres_fwd_kernel(AttnresParams p) {
  constexpr int N = Vec<IO>::N;
  __shared__ float red[AR_MAXW * 2 * AR_MAXS], tot[2 * AR_MAXS], al[AR_MAXS];
  const long long t = blockIdx.x;
  const int S = p.S, d = p.dim, nch = d / N;
  float acc[2 * AR_MAXS];
#pragma unroll
  for (int i = 0; i < 2 * AR_MAXS; ++i) acc[i] = 0.f;
  for (int c = threadIdx.x; c < nch; c += blockDim.x) {
    float w[N], x[N];
#pragma unroll
    for (int e = 0; e < N; ++e) w[e] = p.w[c * N + e];
#pragma unroll
    for (int i = 0; i < AR_MAXS; ++i)
      if (i < S) {
        Vec<IO>::load(static_cast<const IO *>(p.src[i]) + t * d + c * N, x);
#pragma unroll
        for (int e = 0; e < N; ++e) {
          acc[2 * i] = fmaf(x[e], x[e], acc[2 * i]);
          acc[2 * i + 1] = fmaf(w[e], x[e], acc[2 * i + 1]);
        }
      }
  }
  block_sum(acc, 2 * S, red, tot);
  if (threadIdx.x == 0) {
    float lg[AR_MAXS], mx = -INFINITY;
    for (int i = 0; i < S; ++i) {
      const float r = rsqrtf(tot[2 * i] / d + p.eps);
      lg[i] = r * tot[2 * i + 1];
      mx = fmaxf(mx, lg[i]);
      p.rstd[t * S + i] = r;
      p.logit[t * S + i] = lg[i];
    }
    float z = 0.f;
    for (int i = 0; i < S; ++i) {
      lg[i] = __expf(lg[i] - mx);
      z += lg[i];
    }
    for (int i = 0; i < S; ++i) {
      al[i] = lg[i] / z;
      p.alpha[t * S + i] = al[i];
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < nch; c += blockDim.x) {
    float o[N], x[N];
#pragma unroll
    for (int e = 0; e < N; ++e) o[e] = 0.f;
#pragma unroll
    for (int i = 0; i < AR_MAXS; ++i)
      if (i < S) {
        Vec<IO>::load(static_cast<const IO *>(p.src[i]) + t * d + c * N, x);
#pragma unroll
        for (int e = 0; e < N; ++e) o[e] = fmaf(al[i], x[e], o[e]);
      }
    Vec<IO>::store(static_cast<IO *>(p.out) + t * d + c * N, o);
  }
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
  const int threads = ar_threads(p.dim / (f32 ? 4 : 8));
  if (f32)
    attnres_fwd_kernel<float><<<(unsigned)p.T, threads, 0, s>>>(p);
  else
    attnres_fwd_kernel<bf16><<<(unsigned)p.T, threads, 0, s>>>(p);
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
