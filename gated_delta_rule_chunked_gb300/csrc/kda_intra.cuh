// kda_intra.cuh -- intra-chunk building blocks shared by the forward prep kernel
// and the backward's chunk-local gradient kernel: loading a chunk, the Q/K L2
// norms, the per-channel gate scan, the bounded gating factors, the gated Gram
// products and the WY/UT triangular solve.
//
// Gating factorisation. exp(G_r - G_j) is split into two bounded factors so the
// Gram products run as plain matrix multiplies. With 16-token sub-blocks and
// E_a = G at the last row of sub-block a (E_-1 = 0), for r in sub-block a and j
// in sub-block b <= a:
//   exp(G_r - G_j) = exp(G_r - E_{a-1}) * exp(E_{a-1} - G_j)
// The left factor is <= 1. The right factor is <= 1 for b < a, and for b = a it
// is bounded by exp(-(sum of g over that sub-block)), which the library's
// precondition (16-token gate sums >= -80) keeps finite in fp32 and bf16.
#pragma once
#include "kda_common.cuh"

namespace kda {

// ------------------------------------------------------------ shared pieces
// Pair index of sub-block pair (a, b), b <= a: rows [16p, 16p+16) of the RD tile.
__host__ __device__ constexpr int pair_idx(int a, int b) { return a * (a + 1) / 2 + b; }
constexpr int NPAIR = 10;

template <typename E>
struct PrepSmem {
  // byte offsets inside dynamic shared memory
  static constexpr int T128 = 64 * 128 * (int)sizeof(E);
  static constexpr int Q = 0;                       // raw q -> QL -> Qt
  static constexpr int K = Q + T128;                // raw k -> KL -> Kt
  static constexpr int G = K + T128;                // g -> G (log2) ; later A, T (fp32 64x64)
  static constexpr int RD = G + 64 * 128 * 4;       // 10 x 16 rows x 128 (pairs); rows 96.. -> Kh
  static constexpr int VEC = RD + NPAIR * 16 * 128 * (int)sizeof(E);
  // vectors (fp32): rq[64] rk[64] beta[64] E[5][128] gC[128] P[4][128] F[128]
  static constexpr int RQ = VEC, RK = RQ + 256, BETA = RK + 256, EV = BETA + 256, GC = EV + 5 * 512;
  static constexpr int PV = GC + 512, FV = PV + 4 * 512, RQ0 = FV + 512;
  static constexpr int BYTES = RQ0 + 256;
  // aliases after the Gram products
  static constexpr int A = G, T = G + 64 * 64 * 4;  // fp32 [64][64] each
  static constexpr int BM = RD, TB = RD + 64 * 64 * (int)sizeof(E);   // E [64][64] each
  static constexpr int SCR = TB + 64 * 64 * (int)sizeof(E);          // 4 KB solver scratch
  static_assert(SCR + 4096 <= RD + 96 * 128 * (int)sizeof(E), "aliases overlap the Kh rows");
};

// Load raw q, k (E) and g (fp32) rows of one chunk into swizzled tiles; zero past len.
template <typename E>
__device__ __forceinline__ void load_chunk_qkg(char *smem, const E *q, const E *k, const float *g,
                                               const float *beta, long long t0, int len, int h, int H,
                                               int nthreads) {
  using S = PrepSmem<E>;
  Tile<E, 128> tq((E *)(smem + S::Q)), tk((E *)(smem + S::K));
  Tile<float, 128> tg((float *)(smem + S::G));
  constexpr int EPC = 16 / sizeof(E);
  const int tid = threadIdx.x;
  for (int idx = tid; idx < 64 * (128 / EPC); idx += nthreads) {
    const int r = idx / (128 / EPC), ch = idx % (128 / EPC);
    uint4 a = make_uint4(0, 0, 0, 0), b = a;
    if (r < len) {
      const size_t off = ((size_t)(t0 + r) * H + h) * D + ch * EPC;
      a = __ldg(reinterpret_cast<const uint4 *>(q + off));
      b = __ldg(reinterpret_cast<const uint4 *>(k + off));
    }
    *reinterpret_cast<uint4 *>(tq.at(r, ch * EPC)) = a;
    *reinterpret_cast<uint4 *>(tk.at(r, ch * EPC)) = b;
  }
  for (int idx = tid; idx < 64 * 32; idx += nthreads) {
    const int r = idx / 32, ch = idx % 32;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < len) a = __ldg(reinterpret_cast<const float4 *>(g + ((size_t)(t0 + r) * H + h) * D + ch * 4));
    *reinterpret_cast<float4 *>(tg.at(r, ch * 4)) = a;
  }
  float *sb = (float *)(smem + S::BETA);
  for (int r = tid; r < 64; r += nthreads) sb[r] = r < len ? beta[(size_t)(t0 + r) * H + h] : 0.f;
}

// Row norms: rq[r] = scale / sqrt(|q_r|^2 + eps), rk[r] = 1 / sqrt(|k_r|^2 + eps).
// Requires nthreads >= 128 (2 threads per row).
template <typename E>
__device__ __forceinline__ void row_norms(char *smem, float scale) {
  using S = PrepSmem<E>;
  Tile<E, 128> tq((E *)(smem + S::Q)), tk((E *)(smem + S::K));
  const int tid = threadIdx.x;
  if (tid < 128) {
    const int r = tid >> 1, c0 = (tid & 1) * 64;
    float sq = 0.f, sk = 0.f;
#pragma unroll 8
    for (int c = 0; c < 64; ++c) {
      const float a = to_f(*tq.at(r, c0 + c)), b = to_f(*tk.at(r, c0 + c));
      sq = fmaf(a, a, sq);
      sk = fmaf(b, b, sk);
    }
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
    if ((tid & 1) == 0) {
      const float r0 = rsqrtf(sq + 1e-6f);
      ((float *)(smem + S::RQ0))[r] = r0;
      ((float *)(smem + S::RQ))[r] = scale * r0;
      ((float *)(smem + S::RK))[r] = rsqrtf(sk + 1e-6f);
    }
  }
}

// Gate scan (thread c = channel): G (log2 units) in place, E_a into EV.
template <typename E>
__device__ __forceinline__ void gate_scan(char *smem) {
  using S = PrepSmem<E>;
  Tile<float, 128> tg((float *)(smem + S::G));
  float(*ev)[128] = (float(*)[128])(smem + S::EV);
  const int c = threadIdx.x;
  if (c < 128) {
    float run = 0.f;
    ev[0][c] = 0.f;
#pragma unroll 4
    for (int r = 0; r < 64; ++r) {
      run += *tg.at(r, c) * LOG2E;
      *tg.at(r, c) = run;
      if ((r & 15) == 15) ev[1 + (r >> 4)][c] = run;
    }
  }
}

// Factor pass (thread c = channel): QL = q^ x, KL = k^ x (in place), RD pairs.
//   x_r = 2^(G_r - E_{a-1}) <= 1, y_r = 2^(E_a - G_r) <= 1,
//   RD(a', a)[r] = k^_r y_r 2^(E_{a'-1} - E_a)  for a' >= a.
template <typename E>
__device__ __forceinline__ void factor_pass(char *smem) {
  using S = PrepSmem<E>;
  Tile<E, 128> tq((E *)(smem + S::Q)), tk((E *)(smem + S::K));
  Tile<float, 128> tg((float *)(smem + S::G));
  Tile<E, 128> trd((E *)(smem + S::RD));
  const float(*ev)[128] = (const float(*)[128])(smem + S::EV);
  const float *rq = (const float *)(smem + S::RQ), *rk = (const float *)(smem + S::RK);
  const int c = threadIdx.x;
  if (c >= 128) return;
  float e[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) e[i] = ev[i][c];   // e[a+1] = E_a, e[0] = 0
  // per-channel factors used after the Gram products
  float(*pv)[128] = (float(*)[128])(smem + S::PV);
#pragma unroll
  for (int a = 0; a < NSUB; ++a) pv[a][c] = exp2f(e[a]);          // 2^E_{a-1}
  ((float *)(smem + S::FV))[c] = exp2f(e[4] - e[3]);               // 2^(E_3 - E_2)
  ((float *)(smem + S::GC))[c] = exp2f(e[4]);                      // 2^E_3 = exp(G_last)
#pragma unroll
  for (int a = 0; a < NSUB; ++a) {
    float dd[NSUB];
#pragma unroll
    for (int ap = 0; ap < NSUB; ++ap) dd[ap] = ap >= a ? exp2f(e[ap] - e[a + 1]) : 0.f;
#pragma unroll 4
    for (int i = 0; i < SUB; ++i) {
      const int r = a * SUB + i;
      const float Gr = *tg.at(r, c);
      const float x = exp2f(Gr - e[a]), y = exp2f(e[a + 1] - Gr);
      const float kh = to_f(*tk.at(r, c)) * rk[r], qh = to_f(*tq.at(r, c)) * rq[r];
      *tq.at(r, c) = from_f<E>(qh * x);
      *tk.at(r, c) = from_f<E>(kh * x);
      const float ky = kh * y;
#pragma unroll
      for (int ap = a; ap < NSUB; ++ap) *trd.at(pair_idx(ap, a) * SUB + i, c) = from_f<E>(ky * dd[ap]);
    }
  }
}

// Gated Gram products for row sub-block a' = warp (4 warps), kept in registers:
// accA[b][2][4], accB[b][2][4] for column sub-blocks b <= a'.
template <typename E>
__device__ __forceinline__ void gram(char *smem, int ap, float (&accA)[NSUB][2][4], float (&accB)[NSUB][2][4]) {
  using S = PrepSmem<E>;
  Tile<E, 128> tq((E *)(smem + S::Q)), tk((E *)(smem + S::K));
#pragma unroll
  for (int b = 0; b < NSUB; ++b) {
    zero(accA[b]);
    zero(accB[b]);
    if (b <= ap) {
      Tile<E, 128> rd((E *)(smem + S::RD) + pair_idx(ap, b) * SUB * 128);
      wgemm<true, true, 2>(accA[b], tk, ap * SUB, rd, 0, 0, 128);
      wgemm<true, true, 2>(accB[b], tq, ap * SUB, rd, 0, 0, 128);
    }
  }
}

// Solve T = (I + Lm)^-1 for strictly lower Lm (fp32 [64][64] tiles), 4 warps.
__device__ __forceinline__ void ut_solve(float *Lm_p, float *T_p, float *scratch) {
  Tile<float, 64> Lm(Lm_p), T(T_p);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // diagonal 16x16 blocks by forward substitution, one column per lane
  if (warp < NSUB) {
    const int a = warp, j = lane & 15;
    float x[SUB];
#pragma unroll
    for (int i = 0; i < SUB; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
    for (int i = 1; i < SUB; ++i) {
      float s = 0.f;
#pragma unroll
      for (int m = 0; m < i; ++m) s = fmaf(*Lm.at(a * SUB + i, a * SUB + m), x[m], s);
      if (i > j) x[i] = -s;
    }
    if (lane < SUB) {
#pragma unroll
      for (int i = 0; i < SUB; ++i) *T.at(a * SUB + i, a * SUB + j) = x[i];
    }
    // zero the blocks above the diagonal in this block row
    for (int idx = lane; idx < SUB * 64; idx += 32) {
      const int i = idx / 64, cc = idx % 64;
      if (cc >= (a + 1) * SUB) *T.at(a * SUB + i, cc) = 0.f;
    }
  }
  __syncthreads();
  // off-diagonal blocks by levels: T_ab = -T_aa * sum_{m=b}^{a-1} Lm_am T_mb
  float *P = scratch + warp * 256;   // 16x16 per warp
  for (int d = 1; d < NSUB; ++d) {
    const int b = warp, a = warp + d;
    if (a < NSUB) {
      const int i = lane >> 1, j0 = (lane & 1) * 8;
      float acc[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) acc[jj] = 0.f;
      for (int m = b; m < a; ++m) {
#pragma unroll 4
        for (int kk = 0; kk < SUB; ++kk) {
          const float l = *Lm.at(a * SUB + i, m * SUB + kk);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) acc[jj] = fmaf(l, *T.at(m * SUB + kk, b * SUB + j0 + jj), acc[jj]);
        }
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) P[i * 16 + j0 + jj] = acc[jj];
      __syncwarp();
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) acc[jj] = 0.f;
#pragma unroll 4
      for (int kk = 0; kk < SUB; ++kk) {
        const float t = *T.at(a * SUB + i, a * SUB + kk);
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) acc[jj] = fmaf(t, P[kk * 16 + j0 + jj], acc[jj]);
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) *T.at(a * SUB + i, b * SUB + j0 + jj) = -acc[jj];
      __syncwarp();
    }
    __syncthreads();
  }
}

}  // namespace kda
