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

// Sum `n` per-thread values over the CTA (fixed order); results in out[0..n), written by threads
// 0..n-1. There is no barrier after those writes: both callers follow with a cluster barrier
// (release/acquire over every thread of the cluster), which orders them for every reader.
// Inside a warp the values are padded to NP (a power of two) and reduced by recursive halving:
// at each of the first log2(NP) steps a lane sends half of its values to its partner and keeps
// the other half, so after them lane l holds the warp's partial of value idx(l) (one shuffle
// per value kept: NP - 1 in all, instead of 5 per value).
template <int NMAX>
__device__ __forceinline__ void block_sum(float (&v)[NMAX], int n, float *red, float *out) {
  constexpr int NP = NMAX <= 8 ? 8 : (NMAX <= 16 ? 16 : 32);
  constexpr int LG = NP == 8 ? 3 : (NP == 16 ? 4 : 5);   // halving steps
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  float x[NP];
#pragma unroll
  for (int i = 0; i < NP; ++i) x[i] = i < NMAX && i < n ? v[i < NMAX ? i : 0] : 0.f;
  int idx = 0;   // which value this lane ends up holding
#pragma unroll
  for (int st = 0; st < 5; ++st) {
    const int o = 16 >> st;
    if (st < LG) {
      const int half = NP >> (st + 1);
      const bool up = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < half; ++i) {
        const float send = up ? x[i] : x[i + half], keep = up ? x[i + half] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
      if (up) idx += half;
    } else {
      x[0] += __shfl_xor_sync(0xffffffffu, x[0], o);
    }
  }
  if (idx < n && (lane & ((1 << (5 - LG)) - 1)) == 0) red[warp * NMAX + idx] = x[0];
  __syncthreads();
  if ((int)threadIdx.x < n) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += red[w * NMAX + threadIdx.x];
    out[threadIdx.x] = s;
  }
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
// Arrival that publishes nothing (this CTA only signals that its reads of the peers' sums are
// done; their values are already in registers and used), so it needs no release fence.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
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
  } else if ((int)threadIdx.x <= S && nown > 0 && p.prefetch_dist > 0 &&
             (long long)blockIdx.x + p.prefetch_dist < (long long)gridDim.x) {
    // the same quarter of a later token (the distance is a whole number of clusters) into L2,
    // so that CTA's copies hit L2
    const long long t2 = ((long long)blockIdx.x + p.prefetch_dist) / AR_CL;
    prefetch_l2(static_cast<const IO *>(p.src[threadIdx.x - 1]) + t2 * d + (size_t)cbeg * N, (uint32_t)(nown * 16));
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
  cluster_arrive_relaxed();   // done reading the peers' sums; the matching wait comes before exit
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

// Persistent clusters: cluster k of K takes tokens k, k + K, ...; CTA q of the cluster owns
// channel chunks [q per, (q+1) per) (a thread chunks tid + blockDim j, j < J). Per token the
// S source slices and the d_out slice are staged by bulk copies, double-buffered (the next
// token's copies land while this one is computed); pass 1 sums g . x_i over the quarter and
// the cluster adds the four partial sums through distributed shared memory (rank order);
// pass 2 writes dx_i and accumulates the quarter's dw in registers; partial[k][c] at the end.
template <typename IO, int J>
__global__ void __cluster_dims__(AR_CL, 1, 1) __launch_bounds__(256) attnres_bwd_kernel(AttnresParams p) {
  constexpr int N = Vec<IO>::N;
  extern __shared__ __align__(128) char ar_smem[];
  __shared__ float red[8 * AR_MAXS], part[AR_MAXS], st[3][AR_MAXS], dl[AR_MAXS];
  __shared__ __align__(8) uint64_t bar[2];
  const int tid = threadIdx.x;
  const uint32_t q = cluster_rank();
  const long long K = gridDim.x / AR_CL, kc = blockIdx.x / AR_CL;
  const int S = p.S, d = p.dim, nch = d / N, per = (nch + AR_CL - 1) / AR_CL;
  const int cbeg = (int)q * per, cend = min(cbeg + per, nch), nown = max(cend - cbeg, 0);
  const size_t slab = (size_t)(S + 1) * per;   // 16-byte chunks per buffer: S sources, then d_out
  uint4 *buf = reinterpret_cast<uint4 *>(ar_smem);
  const float inv_d = 1.f / d;
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](long long t, int b) {   // thread 0
    fence_proxy_async();
    mbar_expect_tx(&bar[b], (uint32_t)((S + 1) * nown * 16));
    if (nown > 0) {
      for (int i = 0; i < S; ++i)
        bulk_g2s(buf + b * slab + (size_t)i * per, static_cast<const IO *>(p.src[i]) + t * d + (size_t)cbeg * N,
                 (uint32_t)(nown * 16), &bar[b]);
      bulk_g2s(buf + b * slab + (size_t)S * per, static_cast<const IO *>(p.dout) + t * d + (size_t)cbeg * N,
               (uint32_t)(nown * 16), &bar[b]);
    }
  };
  float w[J][N], dwa[J][N];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int c = tid + blockDim.x * j;
#pragma unroll
    for (int e = 0; e < N; ++e) {
      w[j][e] = c < nown ? p.w[(cbeg + c) * N + e] : 0.f;
      dwa[j][e] = 0.f;
    }
  }
  const bool dbl = p.nbuf == 2;   // one buffer when two do not fit: the copies then wait for the previous token
  if (tid == 0 && dbl && kc < p.T) issue(kc, 0);
  bool ok_all = true;
  int it = 0;
  for (long long t = kc; t < p.T; t += K, ++it) {
    const int b = dbl ? (it & 1) : 0;
    __syncthreads();   // the buffer being refilled (the previous token's) and st, dl are consumed
    if (tid == 0) {
      if (!dbl) issue(t, 0);
      else if (t + K < p.T) issue(t + K, b ^ 1);
    } else if (tid <= S + 1 && nown > 0 && t + (dbl ? 2 : 1) * K < p.T) {
      // the slices of the token after the one being copied, into L2: its copies then hit L2
      const long long t2 = t + (dbl ? 2 : 1) * K;
      const void *base = tid <= S ? p.src[tid - 1] : p.dout;
      prefetch_l2(static_cast<const IO *>(base) + t2 * d + (size_t)cbeg * N, (uint32_t)(nown * 16));
    }
    if (tid < S) {
      st[0][tid] = p.alpha[t * S + tid];
      st[1][tid] = p.rstd[t * S + tid];
      st[2][tid] = p.logit[t * S + tid];
    }
    ok_all &= mbar_wait(&bar[b], (uint32_t)((dbl ? it >> 1 : it) & 1));   // on a timeout carry on: the cluster barriers must be met
    const uint4 *xb = buf + b * slab;
    // pass 1: this quarter's g . x_i
    float da[AR_MAXS];
#pragma unroll
    for (int i = 0; i < AR_MAXS; ++i) da[i] = 0.f;
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = tid + blockDim.x * j;
      if (c < nown) {
        float g[N], x[N];
        Vec<IO>::unpack(xb[(size_t)S * per + c], g);
#pragma unroll
        for (int i = 0; i < AR_MAXS; ++i)
          if (i < S) {
            Vec<IO>::unpack(xb[(size_t)i * per + c], x);
#pragma unroll
            for (int e = 0; e < N; ++e) da[i] = fmaf(g[e], x[e], da[i]);
          }
      }
    }
    block_sum(da, S, red, part);
    cluster_arrive();
    cluster_wait();
    if (tid < 32) {   // lane i: the token's g . x_i, then dlogit_i = alpha_i (g . x_i - sum_j alpha_j g . x_j)
      float v = 0.f;
      if (tid < S)
#pragma unroll
        for (uint32_t r = 0; r < AR_CL; ++r) v += ld_peer(&part[tid], r);
      const float a = tid < S ? st[0][tid] : 0.f;
      float m = a * v;
#pragma unroll
      for (int o = 16; o; o >>= 1) m += __shfl_xor_sync(0xffffffffu, m, o);
      if (tid < S) dl[tid] = a * (v - m);
    }
    cluster_arrive_relaxed();   // done reading the peers' sums
    __syncthreads();            // dl
    // pass 2: dx_i and the dw partials
#pragma unroll
    for (int j = 0; j < J; ++j) {
      const int c = tid + blockDim.x * j;
      if (c < nown) {
        float g[N], x[N], dx[N];
        Vec<IO>::unpack(xb[(size_t)S * per + c], g);
#pragma unroll
        for (int i = 0; i < AR_MAXS; ++i)
          if (i < S) {
            Vec<IO>::unpack(xb[(size_t)i * per + c], x);
            const float al = st[0][i], rs = st[1][i], a = rs * dl[i], bb = rs * st[2][i] * inv_d;
#pragma unroll
            for (int e = 0; e < N; ++e) {
              dx[e] = fmaf(al, g[e], a * (w[j][e] - x[e] * bb));
              dwa[j][e] = fmaf(a, x[e], dwa[j][e]);
            }
            Vec<IO>::store(static_cast<IO *>(p.dsrc[i]) + t * d + (size_t)(cbeg + c) * N, dx);
          }
      }
    }
    cluster_wait();   // every peer has read this token's sums before they are rewritten
  }
  if (!ok_all) report(p.status, ERR_TIMEOUT);
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int c = tid + blockDim.x * j;
    if (c < nown)
#pragma unroll
      for (int e = 0; e < N; ++e) p.partial[(size_t)kc * d + (size_t)(cbeg + c) * N + e] = dwa[j][e];
  }
}

__global__ void attnres_dw_reduce_kernel(const float *partial, int nparts, int d, float *dw) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= d) return;
  float s = 0.f;
  for (int b = 0; b < nparts; ++b) s += partial[(size_t)b * d + c];
  dw[c] = s;
}

namespace {
struct BwdShape {
  int per, J, threads, nbuf, smem;
};
BwdShape bwd_shape(bool f32, int dim, int S) {
  BwdShape b;
  b.per = (dim / (f32 ? 4 : 8) + AR_CL - 1) / AR_CL;
  b.J = b.per <= 256 ? 1 : (b.per <= 512 ? 2 : 4);
  b.threads = (b.per + b.J - 1) / b.J;
  b.threads = (b.threads + 31) / 32 * 32;
  if (b.threads < 32) b.threads = 32;
  b.nbuf = 2 * (S + 1) * b.per * 16 <= 200 * 1024 ? 2 : 1;
  b.smem = b.nbuf * (S + 1) * b.per * 16;
  return b;
}
const void *bwd_fn(bool f32, int J) {
  if (f32)
    return J == 1 ? reinterpret_cast<const void *>(attnres_bwd_kernel<float, 1>)
                  : J == 2 ? reinterpret_cast<const void *>(attnres_bwd_kernel<float, 2>)
                           : reinterpret_cast<const void *>(attnres_bwd_kernel<float, 4>);
  return J == 1 ? reinterpret_cast<const void *>(attnres_bwd_kernel<bf16, 1>)
                : J == 2 ? reinterpret_cast<const void *>(attnres_bwd_kernel<bf16, 2>)
                         : reinterpret_cast<const void *>(attnres_bwd_kernel<bf16, 4>);
}
}  // namespace

// Backward clusters: as many as the device holds at once, at most one per token (the dw
// partials are one row per cluster, so this also sizes the workspace).
int attnres_bwd_ctas(long long T, bool f32, int dim, int S) {
  const BwdShape b = bwd_shape(f32, dim, S);
  const void *fn = bwd_fn(f32, b.J);
  int n = 0;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, b.smem) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(AR_CL, 1, 1);
    cfg.blockDim = dim3(b.threads, 1, 1);
    cfg.dynamicSmemBytes = b.smem;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();
  if (n < 1) n = 1;
  return (int)(T < n ? (T > 0 ? T : 1) : n);
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
  // prefetch distance: half the CTAs resident at once, in whole clusters (a quarter to three
  // quarters of a wave measured the same; two waves slower)
  AttnresParams q = p;
  q.prefetch_dist = 0;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) == cudaSuccess)
    q.prefetch_dist = (long long)sms * per_sm / 2 / AR_CL * AR_CL;
  kern<<<grid, threads, smem, s>>>(q);
  return cudaGetLastError();
}

cudaError_t launch_attnres_bwd(const AttnresParams &p, bool f32, cudaStream_t s) {
  const int nparts = attnres_bwd_ctas(p.T, f32, p.dim, p.S);
  if (p.T > 0) {
    const BwdShape b = bwd_shape(f32, p.dim, p.S);
    AttnresParams q = p;
    q.nbuf = b.nbuf;
    void *args[] = {&q};
    cudaError_t e = cudaLaunchKernel(bwd_fn(f32, b.J), dim3((unsigned)(nparts * AR_CL)), dim3(b.threads), args,
                                     (size_t)b.smem, s);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = cudaMemsetAsync(p.partial, 0, (size_t)p.dim * sizeof(float), s);
    if (e != cudaSuccess) return e;
  }
  attnres_dw_reduce_kernel<<<(p.dim + 255) / 256, 256, 0, s>>>(p.partial, nparts, p.dim, p.dw);
  return cudaGetLastError();
}

}  // namespace kda
