// kda_step.cu -- recurrent decode / draft-verify step (memory-bound).
//
// One CTA per (sequence, head). The 128x128 fp32 state (64 KiB) is read once
// into registers (8 warps x 16 rows, each lane 4 consecutive value columns, so
// every row is one coalesced 512-byte float4 access), advanced through the L
// tokens of the call, and written back once -- after accept_len tokens, the
// accepted prefix (ReplaySSM advances KDA state only through accepted tokens:
// "Kimi K3 on Fireworks", rollout section, speculative decoding paragraph).
//
// Per token (gated delta rule, channel-wise decay on the key rows):
//   S' = Diag(exp g) S;  w = S'^T k^;  p = S'^T q^;  u = beta (v - w)
//   S  = S' + k^ u^T;    o = S^T q^ = p + u (k^ . q^)
// The two column reductions w and p share one pass over the state.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int STEP_THREADS = 256;
constexpr int STEP_MAX_L = 8;

template <typename IO>
__device__ __forceinline__ float ld_io(const IO *p) { return to_f(*p); }

template <typename IO>
__device__ __forceinline__ void st_io4(IO *p, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void st_io4<bf16>(bf16 *p, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&lo);
  u.y = *reinterpret_cast<uint32_t *>(&hi);
  *reinterpret_cast<uint2 *>(p) = u;
}
template <>
__device__ __forceinline__ void st_io4<float>(float *p, float a, float b, float c, float d) {
  *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}

template <typename IO>
__global__ void __launch_bounds__(STEP_THREADS, 2) kda_step_kernel(StepParams p) {
  __shared__ float s_q[STEP_MAX_L][D], s_k[STEP_MAX_L][D], s_v[STEP_MAX_L][D], s_dec[STEP_MAX_L][D];
  __shared__ float s_beta[STEP_MAX_L], s_kq[STEP_MAX_L];
  __shared__ __align__(16) float s_red[2][8][2][D];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seq = blockIdx.x / p.heads, h = blockIdx.x % p.heads;
  const int L = p.steps, H = p.heads;
  int acc = p.accept_len ? p.accept_len[seq] : L;
  acc = acc < 0 ? 0 : (acc > L ? L : acc);

  // state rows [16*warp, 16*warp+16), columns [4*lane, 4*lane+4)
  float *st = p.state + ((size_t)seq * H + h) * D * D;
  float4 S[16];
#pragma unroll
  for (int r = 0; r < 16; ++r)
    S[r] = __ldcs(reinterpret_cast<const float4 *>(st + (size_t)(16 * warp + r) * D + 4 * lane));

  // the call's L tokens: raw q, k, v and exp(g) into shared memory
  const IO *q = static_cast<const IO *>(p.q), *k = static_cast<const IO *>(p.k),
           *v = static_cast<const IO *>(p.v);
  for (int idx = tid; idx < L * D; idx += STEP_THREADS) {
    const int l = idx / D, c = idx % D;
    const size_t off = (((size_t)seq * L + l) * H + h) * D + c;
    s_q[l][c] = ld_io(q + off);
    s_k[l][c] = ld_io(k + off);
    s_v[l][c] = ld_io(v + off);
    s_dec[l][c] = __expf(p.g[off]);
  }
  if (tid < L) s_beta[tid] = p.beta[((size_t)seq * L + tid) * H + h];
  __syncthreads();
  // L2 normalisation, one warp per token
  if (warp < L) {
    float sq = 0.f, sk = 0.f, qk = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = s_q[warp][lane + 32 * j], b = s_k[warp][lane + 32 * j];
      sq = fmaf(a, a, sq);
      sk = fmaf(b, b, sk);
      qk = fmaf(a, b, qk);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
      qk += __shfl_xor_sync(0xffffffffu, qk, o);
    }
    const float rq = p.scale * rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      s_q[warp][lane + 32 * j] *= rq;
      s_k[warp][lane + 32 * j] *= rk;
    }
    if (lane == 0) s_kq[warp] = qk * rq * rk;
  }
  __syncthreads();

  IO *o = static_cast<IO *>(p.o);
  for (int l = 0; l < L; ++l) {
    float pw[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int c = 16 * warp + r;
      const float d = s_dec[l][c], kc = s_k[l][c], qc = s_q[l][c];
      S[r].x *= d; S[r].y *= d; S[r].z *= d; S[r].w *= d;
      pw[0] = fmaf(S[r].x, kc, pw[0]); pw[1] = fmaf(S[r].y, kc, pw[1]);
      pw[2] = fmaf(S[r].z, kc, pw[2]); pw[3] = fmaf(S[r].w, kc, pw[3]);
      pq[0] = fmaf(S[r].x, qc, pq[0]); pq[1] = fmaf(S[r].y, qc, pq[1]);
      pq[2] = fmaf(S[r].z, qc, pq[2]); pq[3] = fmaf(S[r].w, qc, pq[3]);
    }
    float(*red)[2][D] = s_red[l & 1];
    *reinterpret_cast<float4 *>(&red[warp][0][4 * lane]) = make_float4(pw[0], pw[1], pw[2], pw[3]);
    *reinterpret_cast<float4 *>(&red[warp][1][4 * lane]) = make_float4(pq[0], pq[1], pq[2], pq[3]);
    __syncthreads();
    float w4[4] = {0.f, 0.f, 0.f, 0.f}, q4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ww = 0; ww < 8; ++ww) {   // fixed order: deterministic
      const float4 a = *reinterpret_cast<const float4 *>(&red[ww][0][4 * lane]);
      const float4 b = *reinterpret_cast<const float4 *>(&red[ww][1][4 * lane]);
      w4[0] += a.x; w4[1] += a.y; w4[2] += a.z; w4[3] += a.w;
      q4[0] += b.x; q4[1] += b.y; q4[2] += b.z; q4[3] += b.w;
    }
    const float beta = s_beta[l], kq = s_kq[l];
    float u[4], out[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      u[j] = beta * (s_v[l][4 * lane + j] - w4[j]);
      out[j] = fmaf(u[j], kq, q4[j]);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const float kc = s_k[l][16 * warp + r];
      S[r].x = fmaf(kc, u[0], S[r].x); S[r].y = fmaf(kc, u[1], S[r].y);
      S[r].z = fmaf(kc, u[2], S[r].z); S[r].w = fmaf(kc, u[3], S[r].w);
    }
    if (warp == 0)
      st_io4<IO>(o + (((size_t)seq * L + l) * H + h) * D + 4 * lane, out[0], out[1], out[2], out[3]);
    if (l + 1 == acc) {
#pragma unroll
      for (int r = 0; r < 16; ++r)
        __stcs(reinterpret_cast<float4 *>(st + (size_t)(16 * warp + r) * D + 4 * lane), S[r]);
    }
  }
}

cudaError_t launch_step(const StepParams &p, bool f32, cudaStream_t s) {
  const unsigned grid = (unsigned)((long long)p.n_seqs * p.heads);
  if (grid == 0) return cudaSuccess;
  if (f32)
    kda_step_kernel<float><<<grid, STEP_THREADS, 0, s>>>(p);
  else
    kda_step_kernel<bf16><<<grid, STEP_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
