// kda_conv.cu -- short causal depthwise convolution on the KDA input side: forward,
// backward and the decode / verify step.
//
//   z[t, c] = bias[c] + sum_{j < W} w[c, j] x[t - (W-1) + j, c],   y = act(z)
// per sequence, positions before its first token read its convolution state (the W - 1
// inputs that preceded it, oldest first). All three kernels are memory-bound streams.
// Forward and backward: a CTA owns a tile of channels (a thread one 16-byte group: 8 bf16
// or 4 fp32; 4 channels in the backward and the step) and a contiguous token range, one CTA
// pair per SM;
// one thread streams the tile's rows into a ring of shared-memory stages with bulk copies
// (up to 96 KB in flight per CTA, independent of registers), every thread walks the rows in
// order keeping the W - 1 previous inputs in registers, so each input row is read from
// memory once (plus W - 1 rows at the range edges) and each output row written once with
// coalesced 16-byte stores.
//
// Backward, with dz = dy act'(z): input row r collects w[c, j] dz[r + (W-1) - j] over the
// taps, dw[c, j] collects dz[t] x[t - (W-1) + j], dbias collects dz; rows before a sequence
// start are the state rows (d_state_in); the gradient of the state after the sequence lands
// on its last W - 1 input rows. A thread sweeps its run plus a W - 1 row halo forward,
// holding the W rows whose sums are still open. dw and dbias are reduced deterministically:
// per-CTA partials over a fixed assignment of runs, then a fixed-order sum.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int CONV_THREADS = 256;
constexpr int CONV_NST = 3;                 // ring stages
constexpr int CONV_STAGE = 32768;           // bytes per stage (all staged tensors of its rows)
constexpr int CONV_SMEM = 128 + CONV_NST * CONV_STAGE;

namespace {

template <typename IO, int V> struct ConvIO;
template <> struct ConvIO<bf16, 8> {
  using Raw = uint4;
  static __device__ __forceinline__ Raw ld(const bf16 *p) { return *reinterpret_cast<const uint4 *>(p); }
  static __device__ __forceinline__ void load(const bf16 *p, float (&f)[8]) { unpack(ld(p), f); }
  static __device__ __forceinline__ void unpack(const uint4 u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[e]));
      f[2 * e] = v.x;
      f[2 * e + 1] = v.y;
    }
  }
  static __device__ __forceinline__ void store(bf16 *p, const float (&f)[8]) {
    uint4 u;
    uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
      w[e] = *reinterpret_cast<const uint32_t *>(&b);
    }
    *reinterpret_cast<uint4 *>(p) = u;
  }
};
template <> struct ConvIO<bf16, 4> {
  using Raw = uint2;
  static __device__ __forceinline__ Raw ld(const bf16 *p) { return *reinterpret_cast<const uint2 *>(p); }
  static __device__ __forceinline__ void load(const bf16 *p, float (&f)[4]) { unpack(ld(p), f); }
  static __device__ __forceinline__ void unpack(const uint2 u, float (&f)[4]) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  }
  static __device__ __forceinline__ void store(bf16 *p, const float (&f)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(f[0], f[1]), b = __floats2bfloat162_rn(f[2], f[3]);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&a);
    u.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
  }
};
template <> struct ConvIO<float, 4> {
  using Raw = float4;
  static __device__ __forceinline__ Raw ld(const float *p) { return *reinterpret_cast<const float4 *>(p); }
  static __device__ __forceinline__ void load(const float *p, float (&f)[4]) { unpack(ld(p), f); }
  static __device__ __forceinline__ void unpack(const float4 v, float (&f)[4]) {
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
  static __device__ __forceinline__ void store(float *p, const float (&f)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};

// Logistic sigmoid. bf16 I/O: one tanh.approx (sigma(z) = (1 + tanh(z / 2)) / 2; the
// instruction's relative error, below 2^-10.9, gives |error| < 2^-11.9 on sigma, under the
// bf16 rounding of the outputs); fp32 I/O: exp and a correctly rounded reciprocal.
template <bool FAST>
__device__ __forceinline__ float sigm(float z) {
  if (FAST) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * z));
    return fmaf(0.5f, t, 0.5f);
  }
  return __frcp_rn(1.f + __expf(-z));
}

// Sequence holding token t (t < T): the last n with cu[n] <= t (skips empty sequences), or
// N equal sequences when cu is NULL.
struct SeqSpan {
  int n;
  long long s0, s1;
};
__device__ __forceinline__ SeqSpan seq_of(const ConvParams &p, long long t) {
  SeqSpan s;
  if (!p.cu) {
    const long long len = p.T / p.n_seqs;
    s.n = (int)(t / len);
    s.s0 = (long long)s.n * len;
    s.s1 = s.s0 + len;
    return s;
  }
  int lo = 0, hi = p.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  s.n = lo;
  s.s0 = p.cu[lo];
  s.s1 = p.cu[lo + 1];
  return s;
}

// Input at token index pos of sequence s (pos >= s0 - (W-1)): a token row, or, before the
// sequence's first token, a row of its state (zero without a state).
template <typename IO, int V, int W>
__device__ __forceinline__ typename ConvIO<IO, V>::Raw input_at(const ConvParams &p, const SeqSpan &s, long long pos,
                                                                int c0) {
  if (pos >= s.s0) return ConvIO<IO, V>::ld(static_cast<const IO *>(p.x) + pos * p.C + c0);
  if (p.st_in) {
    const long long row = (long long)s.n * (W - 1) + (pos - s.s0 + (W - 1));
    return ConvIO<IO, V>::ld(static_cast<const IO *>(p.st_in) + row * p.C + c0);
  }
  typename ConvIO<IO, V>::Raw z;
  memset(&z, 0, sizeof(z));
  return z;
}

// Pre-activation of one token: bias, the current input, then the W - 1 window rows oldest
// first (one order for the forward, the backward's recomputation and the step).
template <typename IO, int V, int W, int WP>
__device__ __forceinline__ void conv_point(const float (&w)[W][V], const float (&b)[V],
                                           const typename ConvIO<IO, V>::Raw (&win)[WP], const float (&xv)[V],
                                           float (&z)[V]) {
#pragma unroll
  for (int e = 0; e < V; ++e) z[e] = fmaf(w[W - 1][e], xv[e], b[e]);
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    float f[V];
    ConvIO<IO, V>::unpack(win[j], f);
#pragma unroll
    for (int e = 0; e < V; ++e) z[e] = fmaf(w[j][e], f[e], z[e]);
  }
}

// Zero-length sequences (only possible with cu): their state passes through unchanged.
// Run by the CTAs of the first token run, for this thread's channels.
template <typename IO, int V, int W>
__device__ void empty_sequences_fwd(const ConvParams &p, int c0) {
  if (!p.cu || !p.st_out || W == 1) return;
  for (int n = 0; n < p.n_seqs; ++n) {
    if (p.cu[n + 1] != p.cu[n]) continue;
#pragma unroll
    for (int i = 0; i < W - 1; ++i) {
      float f[V];
      const long long row = (long long)n * (W - 1) + i;
      if (p.st_in) ConvIO<IO, V>::load(static_cast<const IO *>(p.st_in) + row * p.C + c0, f);
      else
#pragma unroll
        for (int e = 0; e < V; ++e) f[e] = 0.f;
      ConvIO<IO, V>::store(static_cast<IO *>(p.st_out) + row * p.C + c0, f);
    }
  }
}

}  // namespace

namespace {
// Token range [T0, T1) of CTA row `g` out of `G`: whole stages, the remainder to the last rows.
__device__ __forceinline__ void conv_range(long long T, int g, int G, long long &T0, long long &T1) {
  const long long per = (T + G - 1) / G;
  T0 = min((long long)g * per, T);
  T1 = min(T0 + per, T);
}

// Producer side of the ring (thread 0): stage k holds rows [r0 + k ROWS, ...) of `ntens`
// tensors, each row `rowbytes` at src[i] + row * pitch; rows at or past `rend` are not loaded.
template <int ROWS>
__device__ __forceinline__ void conv_issue(char *ring, uint64_t *full, long long k, long long r0, long long rend,
                                           const char *const *src, int ntens, size_t pitch, uint32_t rowbytes) {
  const int slot = (int)(k % CONV_NST);
  const long long a = r0 + k * ROWS;
  const int n = (int)min((long long)ROWS, rend - a);
  if (n <= 0) return;
  fence_proxy_async();   // the threads' reads of this slot come before the copies that refill it
  mbar_expect_tx(&full[slot], (uint32_t)(n * ntens) * rowbytes);
  for (int r = 0; r < n; ++r)
    for (int i = 0; i < ntens; ++i)
      bulk_g2s(ring + (size_t)slot * CONV_STAGE + (size_t)(r * ntens + i) * (CONV_STAGE / (ROWS * ntens)),
               src[i] + (size_t)(a + r) * pitch, rowbytes, &full[slot]);
}

// The rows of stage k into L2 only (a stage beyond the ring, so that its copies hit L2). The
// forward uses it; in the backward (two staged tensors, fp32 dx stores) it measured slower.
template <int ROWS>
__device__ __forceinline__ void conv_prefetch(long long k, long long r0, long long rend, const char *const *src, int ntens,
                                              size_t pitch, uint32_t rowbytes) {
  const long long a = r0 + k * ROWS;
  const int n = (int)min((long long)ROWS, rend - a);
  for (int r = 0; r < n; ++r)
    for (int i = 0; i < ntens; ++i) prefetch_l2(src[i] + (size_t)(a + r) * pitch, rowbytes);
}

// After a wait gave up at stage k: wait (bounded) for the copies of the stages still in flight,
// so none lands after the CTA has left.
__device__ __forceinline__ void conv_drain(uint64_t *full, long long k, long long nst) {
  for (long long j = k + 1; j < k + CONV_NST && j < nst; ++j)
    (void)mbar_wait(&full[j % CONV_NST], (uint32_t)((j / CONV_NST) & 1));
}
}  // namespace

template <typename IO, int W>
__global__ void __launch_bounds__(CONV_THREADS, 2) conv_fwd_kernel(const ConvParams p) {
  constexpr int V = 16 / (int)sizeof(IO);
  constexpr int WP = W > 1 ? W - 1 : 1;
  constexpr bool FAST = sizeof(IO) == 2;
  constexpr int ROWB = CONV_THREADS * V * (int)sizeof(IO);   // 4 KB: one row of the channel tile
  constexpr int ROWS = CONV_STAGE / ROWB;
  using IOV = ConvIO<IO, V>;
  using Raw = typename IOV::Raw;
  extern __shared__ __align__(128) char conv_smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(conv_smem);
  char *ring = conv_smem + 128;
  const int tid = threadIdx.x;
  const int ct0 = blockIdx.x * CONV_THREADS * V;                   // first channel of the tile
  const int nch = min(CONV_THREADS * V, p.C - ct0);
  const bool active = tid * V < nch;
  const int c0 = ct0 + tid * V;
  if (blockIdx.y == 0 && active) empty_sequences_fwd<IO, V, W>(p, c0);
  long long T0, T1;
  conv_range(p.T, blockIdx.y, gridDim.y, T0, T1);
  if (T0 >= T1) return;
  if (tid == 0) {
    for (int i = 0; i < CONV_NST; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const long long nst = (T1 - T0 + ROWS - 1) / ROWS;
  const char *src[1] = {reinterpret_cast<const char *>(static_cast<const IO *>(p.x) + ct0)};
  const size_t pitch = (size_t)p.C * sizeof(IO);
  if (tid == 0)
    for (int k = 0; k < CONV_NST && k < nst; ++k)
      conv_issue<ROWS>(ring, full, k, T0, T1, src, 1, pitch, (uint32_t)(nch * sizeof(IO)));
  float w[W][V], b[V];
  Raw win[WP];   // win[i]: the input at t - (W-1) + i, packed
  SeqSpan s = seq_of(p, T0);
  if (active) {
#pragma unroll
    for (int e = 0; e < V; ++e) {
#pragma unroll
      for (int j = 0; j < W; ++j) w[j][e] = p.w[(size_t)(c0 + e) * W + j];
      b[e] = p.bias ? p.bias[c0 + e] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < W - 1; ++i) win[i] = input_at<IO, V, W>(p, s, T0 - (W - 1) + i, c0);
  }
  for (long long k = 0; k < nst; ++k) {
    const int slot = (int)(k % CONV_NST);
    const bool ok = mbar_wait(&full[slot], (uint32_t)((k / CONV_NST) & 1));
    if (!__syncthreads_and(ok)) {
      if (tid == 0) {
        report(p.status, ERR_TIMEOUT);
        conv_drain(full, k, nst);
      }
      return;
    }
    const char *stage = ring + (size_t)slot * CONV_STAGE + tid * 16;
    const long long tb = T0 + k * ROWS;
    if (active && s.s1 > tb + ROWS && tb + ROWS <= T1) {   // a whole stage inside one sequence, not its last row
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        const long long t = tb + r;
        const Raw xr = *reinterpret_cast<const Raw *>(stage + r * ROWB);
        float xv[V], z[V];
        IOV::unpack(xr, xv);
        conv_point<IO, V, W, WP>(w, b, win, xv, z);
        if (p.act)
#pragma unroll
          for (int e = 0; e < V; ++e) z[e] *= sigm<FAST>(z[e]);
        IOV::store(static_cast<IO *>(p.y) + t * p.C + c0, z);
#pragma unroll
        for (int i = 0; i + 1 < W - 1; ++i) win[i] = win[i + 1];
        if (W > 1) win[WP - 1] = xr;
      }
    } else if (active)
#pragma unroll 4
      for (int r = 0; r < ROWS; ++r) {
        const long long t = tb + r;
        if (t >= T1) break;
        const Raw xr = *reinterpret_cast<const Raw *>(stage + r * ROWB);
        if (t == s.s1) {   // the next (non-empty) sequence starts here: its window is its state
          s = seq_of(p, t);
#pragma unroll
          for (int i = 0; i < W - 1; ++i) win[i] = input_at<IO, V, W>(p, s, t - (W - 1) + i, c0);
        }
        float xv[V], z[V];
        IOV::unpack(xr, xv);
        conv_point<IO, V, W, WP>(w, b, win, xv, z);
        if (p.act)
#pragma unroll
          for (int e = 0; e < V; ++e) z[e] *= sigm<FAST>(z[e]);
        IOV::store(static_cast<IO *>(p.y) + t * p.C + c0, z);
#pragma unroll
        for (int i = 0; i + 1 < W - 1; ++i) win[i] = win[i + 1];
        if (W > 1) win[WP - 1] = xr;
        if (t == s.s1 - 1 && p.st_out)
#pragma unroll
          for (int i = 0; i < W - 1; ++i)
            *reinterpret_cast<Raw *>(static_cast<IO *>(p.st_out) + ((long long)s.n * (W - 1) + i) * p.C + c0) = win[i];
      }
    __syncthreads();   // every thread is done with this slot
    if (tid == 0 && k + CONV_NST < nst) {
      conv_issue<ROWS>(ring, full, k + CONV_NST, T0, T1, src, 1, pitch, (uint32_t)(nch * sizeof(IO)));
      if (k + CONV_NST + 1 < nst) conv_prefetch<ROWS>(k + CONV_NST + 1, T0, T1, src, 1, pitch, (uint32_t)(nch * sizeof(IO)));
    }
  }
}

namespace {
// Backward: one pending row leaves the open window; store it where it belongs.
//   row >= s0:              an input row; stored if this run owns it (t0 <= row < tend)
//   s0 - (W-1) <= row < s0: a state row; stored if this run holds the sequence start
// plus the gradient of the state after the sequence for rows among its last W - 1.
template <int W>
__device__ __forceinline__ void conv_flush(const ConvParams &p, const SeqSpan &s, long long row, long long t0,
                                           long long tend, int c0, const float (&v)[4]) {
  constexpr int V = 4;
  const bool input_row = row >= s.s0;
  if (input_row ? !(row >= t0 && row < tend) : !(row >= s.s0 - (W - 1) && s.s0 >= t0 && p.dst)) return;
  float o[V];
#pragma unroll
  for (int e = 0; e < V; ++e) o[e] = v[e];
  if (p.dso && W > 1 && row >= s.s1 - (W - 1)) {
    const float4 d =
        *reinterpret_cast<const float4 *>(p.dso + ((long long)s.n * (W - 1) + (row - (s.s1 - (W - 1)))) * p.C + c0);
    o[0] += d.x; o[1] += d.y; o[2] += d.z; o[3] += d.w;
  }
  float *dst = input_row ? p.dx + row * p.C + c0 : p.dst + ((long long)s.n * (W - 1) + (row - s.s0 + (W - 1))) * p.C + c0;
  *reinterpret_cast<float4 *>(dst) = make_float4(o[0], o[1], o[2], o[3]);
}
}  // namespace

template <typename IO, int W>
__global__ void __launch_bounds__(CONV_THREADS, 2) conv_bwd_kernel(const ConvParams p) {
  constexpr int V = 4;
  constexpr int WP = W > 1 ? W - 1 : 1;
  constexpr bool FAST = sizeof(IO) == 2;
  constexpr int ROWB = CONV_THREADS * V * (int)sizeof(IO);   // one row of one tensor of the tile
  constexpr int ROWS = CONV_STAGE / (2 * ROWB);               // x and dy rows per stage
  using IOV = ConvIO<IO, V>;
  using Raw = typename IOV::Raw;
  extern __shared__ __align__(128) char conv_smem[];
  uint64_t *full = reinterpret_cast<uint64_t *>(conv_smem);
  char *ring = conv_smem + 128;
  const int tid = threadIdx.x;
  const int ct0 = blockIdx.x * CONV_THREADS * V;
  const int nch = min(CONV_THREADS * V, p.C - ct0);
  const bool active = tid * V < nch;
  const int c0 = ct0 + tid * V;
  if (blockIdx.y == 0 && active && p.cu && p.dst && W > 1)   // zero-length sequences: d_state_in = d_state_out
    for (int n = 0; n < p.n_seqs; ++n) {
      if (p.cu[n + 1] != p.cu[n]) continue;
      for (int i = 0; i < W - 1; ++i) {
        const long long off = ((long long)n * (W - 1) + i) * p.C + c0;
        *reinterpret_cast<float4 *>(p.dst + off) =
            p.dso ? *reinterpret_cast<const float4 *>(p.dso + off) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  float dwp[W][V], dbp[V];
#pragma unroll
  for (int e = 0; e < V; ++e) {
#pragma unroll
    for (int j = 0; j < W; ++j) dwp[j][e] = 0.f;
    dbp[e] = 0.f;
  }
  long long T0, T1;
  conv_range(p.T, blockIdx.y, gridDim.y, T0, T1);
  if (T0 < T1) {
    const long long thalo = min(T1 + (W - 1), p.T);
    if (tid == 0) {
      for (int i = 0; i < CONV_NST; ++i) mbar_init(&full[i], 1);
      fence_mbar_init();
    }
    __syncthreads();
    const long long nst = (thalo - T0 + ROWS - 1) / ROWS;
    const char *src[2] = {reinterpret_cast<const char *>(static_cast<const IO *>(p.x) + ct0),
                          reinterpret_cast<const char *>(static_cast<const IO *>(p.dy) + ct0)};
    const size_t pitch = (size_t)p.C * sizeof(IO);
    const uint32_t rowbytes = (uint32_t)(nch * sizeof(IO));
    if (tid == 0)
      for (int k = 0; k < CONV_NST && k < nst; ++k) conv_issue<ROWS>(ring, full, k, T0, thalo, src, 2, pitch, rowbytes);
    float w[W][V], b[V];
    Raw win[WP];
    float pend[W][V];   // pend[m]: open sum of row t - m
    SeqSpan s = seq_of(p, T0);
    if (active) {
#pragma unroll
      for (int e = 0; e < V; ++e) {
#pragma unroll
        for (int j = 0; j < W; ++j) w[j][e] = p.w[(size_t)(c0 + e) * W + j];
        b[e] = p.bias ? p.bias[c0 + e] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < W - 1; ++i) win[i] = input_at<IO, V, W>(p, s, T0 - (W - 1) + i, c0);
    }
#pragma unroll
    for (int m = 0; m < W; ++m)
#pragma unroll
      for (int e = 0; e < V; ++e) pend[m][e] = 0.f;
    bool done = false;   // the sweep met the start of a sequence this range does not own
    for (long long k = 0; k < nst; ++k) {
      const int slot = (int)(k % CONV_NST);
      const bool ok = mbar_wait(&full[slot], (uint32_t)((k / CONV_NST) & 1));
      if (!__syncthreads_and(ok)) {
        if (tid == 0) {
          report(p.status, ERR_TIMEOUT);
          conv_drain(full, k, nst);
        }
        return;
      }
      const char *stage = ring + (size_t)slot * CONV_STAGE + tid * V * (int)sizeof(IO);
      const long long tb = T0 + k * ROWS;
      // a stage inside one sequence and inside the range, away from its edges: every row is
      // owned, every row leaving the window is an owned input row with no state-out gradient
      const bool plain = s.s1 >= tb + ROWS && tb + ROWS <= T1 && tb - W >= T0 && tb - W >= s.s0;
      if (active && !done && plain) {
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
          const long long t = tb + r;
          const Raw xr = *reinterpret_cast<const Raw *>(stage + (2 * r) * ROWB);
          const Raw gr = *reinterpret_cast<const Raw *>(stage + (2 * r + 1) * ROWB);
          *reinterpret_cast<float4 *>(p.dx + (t - W) * p.C + c0) =
              make_float4(pend[W - 1][0], pend[W - 1][1], pend[W - 1][2], pend[W - 1][3]);
#pragma unroll
          for (int m = W - 1; m > 0; --m)
#pragma unroll
            for (int e = 0; e < V; ++e) pend[m][e] = pend[m - 1][e];
          float xv[V], gv[V], wf[WP][V], z[V], dz[V];
          IOV::unpack(xr, xv);
          IOV::unpack(gr, gv);
#pragma unroll
          for (int j = 0; j < W - 1; ++j) IOV::unpack(win[j], wf[j]);
#pragma unroll
          for (int e = 0; e < V; ++e) {
            z[e] = fmaf(w[W - 1][e], xv[e], b[e]);
#pragma unroll
            for (int j = 0; j < W - 1; ++j) z[e] = fmaf(w[j][e], wf[j][e], z[e]);
            if (p.act) {
              const float sg = sigm<FAST>(z[e]);
              dz[e] = gv[e] * sg * fmaf(z[e], 1.f - sg, 1.f);
            } else {
              dz[e] = gv[e];
            }
            pend[0][e] = w[W - 1][e] * dz[e];
#pragma unroll
            for (int m = 1; m < W; ++m) pend[m][e] = fmaf(w[W - 1 - m][e], dz[e], pend[m][e]);
            dbp[e] += dz[e];
            dwp[W - 1][e] = fmaf(dz[e], xv[e], dwp[W - 1][e]);
#pragma unroll
            for (int j = 0; j < W - 1; ++j) dwp[j][e] = fmaf(dz[e], wf[j][e], dwp[j][e]);
          }
#pragma unroll
          for (int i = 0; i + 1 < W - 1; ++i) win[i] = win[i + 1];
          if (W > 1) win[WP - 1] = xr;
        }
      } else if (active && !done)
#pragma unroll 2
        for (int r = 0; r < ROWS; ++r) {
          const long long t = tb + r;
          if (t >= thalo) break;
          const Raw xr = *reinterpret_cast<const Raw *>(stage + (2 * r) * ROWB);
          const Raw gr = *reinterpret_cast<const Raw *>(stage + (2 * r + 1) * ROWB);
          if (t == s.s1) {   // sequence end: close its open rows
#pragma unroll
            for (int m = 0; m < W; ++m) conv_flush<W>(p, s, t - 1 - m, T0, T1, c0, pend[m]);
            if (t >= T1) {   // the next sequence belongs to the next range
              done = true;
              break;
            }
            s = seq_of(p, t);
#pragma unroll
            for (int i = 0; i < W - 1; ++i) win[i] = input_at<IO, V, W>(p, s, t - (W - 1) + i, c0);
#pragma unroll
            for (int m = 0; m < W; ++m)
#pragma unroll
              for (int e = 0; e < V; ++e) pend[m][e] = 0.f;
          }
          // row t - W leaves the window
          conv_flush<W>(p, s, t - W, T0, T1, c0, pend[W - 1]);
#pragma unroll
          for (int m = W - 1; m > 0; --m)
#pragma unroll
            for (int e = 0; e < V; ++e) pend[m][e] = pend[m - 1][e];
          float xv[V], gv[V], z[V];
          IOV::unpack(xr, xv);
          IOV::unpack(gr, gv);
          conv_point<IO, V, W, WP>(w, b, win, xv, z);
          float dz[V];
#pragma unroll
          for (int e = 0; e < V; ++e) {
            if (p.act) {
              const float sg = sigm<FAST>(z[e]);
              dz[e] = gv[e] * sg * fmaf(z[e], 1.f - sg, 1.f);
            } else {
              dz[e] = gv[e];
            }
            pend[0][e] = w[W - 1][e] * dz[e];
#pragma unroll
            for (int m = 1; m < W; ++m) pend[m][e] = fmaf(w[W - 1 - m][e], dz[e], pend[m][e]);
          }
          if (t < T1) {
#pragma unroll
            for (int e = 0; e < V; ++e) {
              dbp[e] += dz[e];
              dwp[W - 1][e] = fmaf(dz[e], xv[e], dwp[W - 1][e]);
            }
#pragma unroll
            for (int j = 0; j < W - 1; ++j) {
              float f[V];
              IOV::unpack(win[j], f);
#pragma unroll
              for (int e = 0; e < V; ++e) dwp[j][e] = fmaf(dz[e], f[e], dwp[j][e]);
            }
          }
#pragma unroll
          for (int i = 0; i + 1 < W - 1; ++i) win[i] = win[i + 1];
          if (W > 1) win[WP - 1] = xr;
        }
      __syncthreads();   // every thread is done with this slot
      if (tid == 0 && k + CONV_NST < nst) conv_issue<ROWS>(ring, full, k + CONV_NST, T0, thalo, src, 2, pitch, rowbytes);
    }
    if (active && !done)   // the sweep reached thalo inside the sequence: close what is open
#pragma unroll
      for (int m = 0; m < W; ++m) conv_flush<W>(p, s, thalo - 1 - m, T0, T1, c0, pend[m]);
  }
  // per-CTA partials: partial[blockIdx.y][c][W + 1] (taps, then the bias)
  if (!active) return;
  float *part = p.partial + ((size_t)blockIdx.y * p.C + c0) * (W + 1);
#pragma unroll
  for (int e = 0; e < V; ++e) {
#pragma unroll
    for (int j = 0; j < W; ++j) part[e * (W + 1) + j] = dwp[j][e];
    part[e * (W + 1) + W] = dbp[e];
  }
}

__global__ void conv_dw_reduce_kernel(const float *partial, int groups, int C, int W, float *dw, float *db) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long n = (long long)C * (W + 1);
  if (i >= n) return;
  float s = 0.f;
  for (int g = 0; g < groups; ++g) s += partial[(size_t)g * n + i];
  const int c = (int)(i / (W + 1)), j = (int)(i % (W + 1));
  if (j < W) dw[(size_t)c * W + j] = s;
  else if (db) db[c] = s;
}

// NS sequences per thread (the weights are loaded once for all of them); LM >= L token slots
// held in registers (1, 2, 4 or 8: fewer registers, more warps per SM for short calls); VW:
// weight and bias rows 16-byte aligned, loaded as float4 (the V x W weights of V consecutive
// channels are contiguous). Every sequence's state rows and token rows are loaded before any
// arithmetic.
template <typename IO, int W, int NS, int LM, bool VW>
__global__ void __launch_bounds__(CONV_THREADS, NS > 1                ? 2
                                                : sizeof(IO) == 2      ? (LM <= 2 ? 6 : LM == 4 ? 5 : 4)
                                                                       : (LM <= 4 ? 3 : 2))
    conv_step_kernel(const ConvParams p) {
  constexpr int V = 4;   // 4 channels a thread: few registers, many warps for a latency-bound call
  constexpr int WP = W > 1 ? W - 1 : 1;
  constexpr bool FAST = sizeof(IO) == 2;
  using IOV = ConvIO<IO, V>;
  using Raw = typename IOV::Raw;
  const int cg = blockIdx.x * CONV_THREADS + threadIdx.x;
  if (p.prefetch_dist > 0 && (int)threadIdx.x < W - 1 + p.L) {
    // the state rows (threads < W - 1) and token rows of the CTA about one wave later into L2
    const long long lin = (long long)blockIdx.y * gridDim.x + blockIdx.x + p.prefetch_dist;
    const int bx = (int)(lin % gridDim.x), n2 = (int)(lin / gridDim.x) * NS;
    const int cb = bx * CONV_THREADS * V, nb = min(CONV_THREADS * V, p.C - cb) * (int)sizeof(IO) / 16 * 16;
    if (lin < (long long)gridDim.x * gridDim.y && n2 < p.n_seqs && nb > 0) {
      const int i = threadIdx.x;
      if (i < W - 1) {
        const int slot = p.idx ? p.idx[n2] : n2;
        if (slot >= 0 && slot < p.n_slots)
          prefetch_l2(static_cast<const IO *>(p.st_out) + ((size_t)slot * (W - 1) + i) * p.C + cb, (uint32_t)nb);
      } else {
        prefetch_l2(static_cast<const IO *>(p.x) + ((size_t)n2 * p.L + (i - (W - 1))) * p.C + cb, (uint32_t)nb);
      }
    }
  }
  if (cg >= p.C / V) return;
  const int c0 = cg * V, L = p.L;
  int F[NS], acc[NS];
  bool live[NS];
  IO *st[NS];
  Raw win[NS][WP], xr[NS][LM];
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    const int n = blockIdx.y * NS + u;
    live[u] = n < p.n_seqs;
    const int slot = !live[u] ? 0 : (p.idx ? p.idx[n] : n);
    if (live[u] && (slot < 0 || slot >= p.n_slots)) {
      if (cg == 0) report(p.status, KDA_ERR_INVALID_ARG_CODE);
      live[u] = false;
    }
    F[u] = live[u] && p.first ? min(max(p.first[n], 0), L) : 0;
    acc[u] = live[u] && p.acc ? min(max(p.acc[n], 0), L) : L;
    st[u] = static_cast<IO *>(p.st_out) + (size_t)slot * (W - 1) * p.C + c0;
    if (live[u]) {
#pragma unroll
      for (int i = 0; i < W - 1; ++i) win[u][i] = IOV::ld(st[u] + (size_t)i * p.C);
#pragma unroll
      for (int l = 0; l < LM; ++l)
        if (l >= F[u] && l < L) xr[u][l] = IOV::ld(static_cast<const IO *>(p.x) + ((size_t)n * L + l) * p.C + c0);
    }
  }
  float w[W][V], b[V];
  if (VW) {
    const float4 *w4 = reinterpret_cast<const float4 *>(p.w + (size_t)c0 * W);
#pragma unroll
    for (int i = 0; i < W; ++i) {   // V * W = 4 W floats
      const float4 t = w4[i];
      const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) w[(4 * i + k) % W][(4 * i + k) / W] = tv[k];
    }
    const float4 t = p.bias ? *reinterpret_cast<const float4 *>(p.bias + c0) : make_float4(0.f, 0.f, 0.f, 0.f);
    b[0] = t.x; b[1] = t.y; b[2] = t.z; b[3] = t.w;
  } else {
#pragma unroll
    for (int e = 0; e < V; ++e) {
#pragma unroll
      for (int j = 0; j < W; ++j) w[j][e] = p.w[(size_t)(c0 + e) * W + j];
      b[e] = p.bias ? p.bias[c0 + e] : 0.f;
    }
  }
#pragma unroll
  for (int u = 0; u < NS; ++u) {
    if (!live[u]) continue;
    const int n = blockIdx.y * NS + u;
    Raw keep[WP];
#pragma unroll
    for (int l = 0; l < LM; ++l) {
      if (l < F[u] || l >= L) continue;
      float xv[V], z[V];
      IOV::unpack(xr[u][l], xv);
      conv_point<IO, V, W, WP>(w, b, win[u], xv, z);
      if (p.act)
#pragma unroll
        for (int e = 0; e < V; ++e) z[e] *= sigm<FAST>(z[e]);
      IOV::store(static_cast<IO *>(p.y) + ((size_t)n * L + l) * p.C + c0, z);
#pragma unroll
      for (int i = 0; i + 1 < W - 1; ++i) win[u][i] = win[u][i + 1];
      if (W > 1) win[u][WP - 1] = xr[u][l];
      if (l + 1 == acc[u])
#pragma unroll
        for (int i = 0; i < W - 1; ++i) keep[i] = win[u][i];
    }
    if (acc[u] > F[u])
#pragma unroll
      for (int i = 0; i < W - 1; ++i) *reinterpret_cast<Raw *>(st[u] + (size_t)i * p.C) = keep[i];
  }
}

namespace {
int sm_count_dev() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0)
    n = 1;
  return n;
}
// CTA rows (token ranges) for `xblocks` channel tiles: two CTAs per SM (96 KB of ring each), one wave.
int conv_rows(int xblocks) {
  const int g = 2 * sm_count_dev() / xblocks;
  return g < 1 ? 1 : (g > 65535 ? 65535 : g);
}
template <typename IO, int W>
cudaError_t fwd_w(const ConvParams &p, cudaStream_t s) {
  constexpr int V = 16 / (int)sizeof(IO);
  const int xb = (p.C / V + CONV_THREADS - 1) / CONV_THREADS;
  cudaError_t e = cudaFuncSetAttribute(conv_fwd_kernel<IO, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, CONV_SMEM);
  if (e != cudaSuccess) return e;
  conv_fwd_kernel<IO, W><<<dim3((unsigned)xb, (unsigned)conv_rows(xb)), CONV_THREADS, CONV_SMEM, s>>>(p);
  return cudaGetLastError();
}
template <typename IO>
cudaError_t fwd_t(const ConvParams &p, cudaStream_t s) {
  switch (p.W) {
    case 1: return fwd_w<IO, 1>(p, s);
    case 2: return fwd_w<IO, 2>(p, s);
    case 3: return fwd_w<IO, 3>(p, s);
    default: return fwd_w<IO, 4>(p, s);
  }
}
template <typename IO, int W>
cudaError_t bwd_w(const ConvParams &p, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(conv_bwd_kernel<IO, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, CONV_SMEM);
  if (e != cudaSuccess) return e;
  conv_bwd_kernel<IO, W><<<dim3((unsigned)((p.C / 4 + CONV_THREADS - 1) / CONV_THREADS), (unsigned)p.groups),
                           CONV_THREADS, CONV_SMEM, s>>>(p);
  return cudaGetLastError();
}
template <typename IO>
cudaError_t bwd_t(const ConvParams &p, cudaStream_t s) {
  switch (p.W) {
    case 1: return bwd_w<IO, 1>(p, s);
    case 2: return bwd_w<IO, 2>(p, s);
    case 3: return bwd_w<IO, 3>(p, s);
    default: return bwd_w<IO, 4>(p, s);
  }
}
constexpr int CONV_STEP_NS = 1;   // sequences per thread
template <typename IO, int W, int LM, bool VW>
void step_v(const ConvParams &p, dim3 grid, cudaStream_t s) {
  auto kern = conv_step_kernel<IO, W, CONV_STEP_NS, LM, VW>;
  // prefetch distance: the CTAs resident at once (one wave); rows must start on 16 bytes
  ConvParams q = p;
  q.prefetch_dist = 0;
  int dev = 0, sms = 0, per_sm = 0;
  if ((size_t)p.C * sizeof(IO) % 16 == 0 && reinterpret_cast<uintptr_t>(p.x) % 16 == 0 &&
      reinterpret_cast<uintptr_t>(p.st_out) % 16 == 0 && cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, CONV_THREADS, 0) == cudaSuccess)
    q.prefetch_dist = (long long)sms * per_sm;
  kern<<<grid, CONV_THREADS, 0, s>>>(q);
}
template <typename IO, int W, int LM>
void step_l(const ConvParams &p, dim3 grid, cudaStream_t s) {
  const bool vw = reinterpret_cast<uintptr_t>(p.w) % 16 == 0 && reinterpret_cast<uintptr_t>(p.bias) % 16 == 0;
  if (vw)
    step_v<IO, W, LM, true>(p, grid, s);
  else
    step_v<IO, W, LM, false>(p, grid, s);
}
template <typename IO, int W>
void step_w(const ConvParams &p, dim3 grid, cudaStream_t s) {
  if (p.L <= 1) step_l<IO, W, 1>(p, grid, s);
  else if (p.L <= 2) step_l<IO, W, 2>(p, grid, s);
  else if (p.L <= 4) step_l<IO, W, 4>(p, grid, s);
  else step_l<IO, W, 8>(p, grid, s);
}
template <typename IO>
cudaError_t step_t(const ConvParams &p, cudaStream_t s) {
  constexpr int V = 4;
  const dim3 grid((unsigned)((p.C / V + CONV_THREADS - 1) / CONV_THREADS),
                  (unsigned)((p.n_seqs + CONV_STEP_NS - 1) / CONV_STEP_NS));
  switch (p.W) {
    case 1: step_w<IO, 1>(p, grid, s); break;
    case 2: step_w<IO, 2>(p, grid, s); break;
    case 3: step_w<IO, 3>(p, grid, s); break;
    default: step_w<IO, 4>(p, grid, s); break;
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_conv_fwd(const ConvParams &p, bool f32, cudaStream_t s) {
  if (p.T == 0) return cudaSuccess;
  return f32 ? fwd_t<float>(p, s) : fwd_t<bf16>(p, s);
}

// Backward CTA rows; the dw partials are per CTA row, so this also sizes the workspace.
int conv_bwd_groups(long long T, int C, int W, bool f32) {
  (void)T;
  (void)W;
  (void)f32;
  return conv_rows((C / 4 + CONV_THREADS - 1) / CONV_THREADS);
}

cudaError_t launch_conv_bwd(const ConvParams &p, bool f32, cudaStream_t s) {
  const long long n = (long long)p.C * (p.W + 1);
  if (p.T > 0) {
    cudaError_t e = f32 ? bwd_t<float>(p, s) : bwd_t<bf16>(p, s);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = cudaMemsetAsync(p.partial, 0, (size_t)n * sizeof(float), s);
    if (e != cudaSuccess) return e;
  }
  conv_dw_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p.partial, p.T > 0 ? p.groups : 1, p.C, p.W, p.dw,
                                                                     p.db);
  return cudaGetLastError();
}

cudaError_t launch_conv_step(const ConvParams &p, bool f32, cudaStream_t s) {
  if (p.n_seqs == 0) return cudaSuccess;
  return f32 ? step_t<float>(p, s) : step_t<bf16>(p, s);
}

}  // namespace kda
