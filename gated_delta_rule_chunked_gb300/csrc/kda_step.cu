// kda_step.cu -- recurrent decode / draft-verify step (memory-bound).
//
// One CTA per (sequence, head). The 128x128 fp32 state S0 (64 KiB) is read
// once into registers (8 warps x 16 key rows, each lane 4 consecutive value
// columns, so every row is one coalesced 512-byte float4 access) and written
// back once, after accept_len tokens -- the accepted prefix (ReplaySSM advances
// KDA state only through accepted tokens: "Kimi K3 on Fireworks", rollout
// section, speculative decoding paragraph).
//
// The L tokens of a call are evaluated against S0 together instead of one at a
// time (the KDA recurrence unrolled over the call). With G_l = g_1 + .. + g_l
// (per key channel), gamma_l = exp(G_l) and the token recurrence
//   S_l = Diag(exp g_l) S_{l-1} + k^_l u_l^T,  u_l = beta_l (v_l - (Diag(exp g_l) S_{l-1})^T k^_l),
//   o_l = S_l^T q^_l,
// every quantity is S0 seen through a decayed vector plus a small coupling
// between the call's own tokens:
//   w_l = S0^T (gamma_l o k^_l) + sum_{m<l} a_lm u_m,   a_lm = sum_c k^_m k^_l exp(G_l - G_m)
//   o_l = S0^T (gamma_l o q^_l) + sum_{m<l} b_lm u_m + (k^_l . q^_l) u_l,
//                                                     b_lm = sum_c k^_m q^_l exp(G_l - G_m)
//   S_A = Diag(gamma_A) S0 + sum_{m<=A} (exp(G_A - G_m) o k^_m) u_m^T   (A = accept_len).
// So the state is swept twice per call (2L column sums, then one rank-A
// update), with one cross-warp reduction, instead of twice per token.
//
// Two-phase draft/verify: the state of a sequence may sit in any slot of a pool
// (state_indices), and a call's leading slots may be padding (first_slot): a
// padded slot stands for zero inputs, beta = 0 and g = 0, which leave S and every
// other token's quantities exactly as they were, so the kernel skips it (its inputs
// are not read, its output is not written). A call
// can thus replay a sequence's accepted draft tokens (right-aligned before the new
// draft) and commit after them while verifying the next draft in the same pass.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int STEP_THREADS = 256;
constexpr int STEP_MAX_L = 8;

__device__ __forceinline__ float2 dup2(float a) { return make_float2(a, a); }

// a 4-byte global -> shared copy that holds no register (cp_async16 is its 16-byte form)
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(__cvta_generic_to_global(src))
               : "memory");
}

// Shared memory of one CTA (static part; the column-sum partials are dynamic).
struct StepSmem {
  float q[STEP_MAX_L][D];    // q^ (times scale)
  float k[STEP_MAX_L][D];    // k^
  float v[STEP_MAX_L][D];
  float G[STEP_MAX_L][D];    // raw g, then the running sums G_l
  float kt[STEP_MAX_L][D];   // gamma_l o k^_l
  float qt[STEP_MAX_L][D];   // gamma_l o q^_l
  float kc[STEP_MAX_L][D];   // exp(G_A - G_m) o k^_m
  float U[STEP_MAX_L][D];    // u_m
  float gA[D];               // gamma_A
  float a[STEP_MAX_L][STEP_MAX_L], b[STEP_MAX_L][STEP_MAX_L];
  float beta[STEP_MAX_L];
};

// PAD: the call has padded leading slots (first_slot given); without them F = 0 is a constant.
template <typename IO, bool PAD>
__global__ void __launch_bounds__(STEP_THREADS, 2) kda_step_kernel(StepParams p) {
  __shared__ __align__(16) StepSmem sm;
  // partials [8 row groups][2L vectors][D]
  extern __shared__ __align__(16) float step_red[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seq = blockIdx.x / p.heads, h = blockIdx.x % p.heads;
  const int LS = p.steps, H = p.heads;   // token slots of the call
  int A = p.accept_len ? p.accept_len[seq] : LS;
  A = A < 0 ? 0 : (A > LS ? LS : A);
  // slots before F are padding: zero inputs, beta = 0 and g = 0 make them exact identities, so
  // only the L = LS - F real slots are evaluated (real token l is slot F + l) and the state is
  // committed after A - F of them
  int F = PAD ? p.first_slot[seq] : 0;
  F = F < 0 ? 0 : (F > LS ? LS : F);
  const int L = LS - F, NV = 2 * L;
  A = A > F ? A - F : 0;
  const int slot = p.state_indices ? p.state_indices[seq] : seq;
  if (p.state_indices && (slot < 0 || slot >= p.n_slots)) {   // block-uniform
    if (tid == 0) report(p.status, KDA_ERR_INVALID_ARG_CODE);
    return;
  }
  if (L == 0) return;   // padding only: no output, the state is unchanged
  float *red = step_red;

  // The call's token rows go straight to shared memory first (q, k, v in the io type into the
  // head of the partials area, free until sweep 1; g into G; beta), so that the state loads
  // below are issued at once and the token work overlaps their arrival.
  const IO *q = static_cast<const IO *>(p.q), *k = static_cast<const IO *>(p.k),
           *v = static_cast<const IO *>(p.v);
  IO *raw = reinterpret_cast<IO *>(step_red);   // [q, k, v][L][D]
  {
    constexpr int CPR = D * (int)sizeof(IO) / 16, CPG = D * (int)sizeof(float) / 16;   // 16-byte pieces per row
    const size_t row0 = ((size_t)seq * LS + F) * H + h;   // token slot F + l is row row0 + l * H
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      const IO *src = a == 0 ? q : a == 1 ? k : v;
      for (int t = tid; t < L * CPR; t += STEP_THREADS) {
        const int l = t / CPR, c = t % CPR;
        cp_async16(reinterpret_cast<char *>(raw + ((size_t)a * L + l) * D) + 16 * c,
                   reinterpret_cast<const char *>(src + (row0 + (size_t)l * H) * D) + 16 * c);
      }
    }
    for (int t = tid; t < L * CPG; t += STEP_THREADS) {
      const int l = t / CPG, c = t % CPG;
      cp_async16(reinterpret_cast<char *>(&sm.G[l][0]) + 16 * c,
                 reinterpret_cast<const char *>(p.g + (row0 + (size_t)l * H) * D) + 16 * c);
    }
    if (tid < L) cp_async4(&sm.beta[tid], p.beta + row0 + (size_t)tid * H);
  }

  // state rows [16 warp, +16), columns [4 lane, +4) as two column pairs
  float *st = p.state + ((size_t)slot * H + h) * D * D;
  float2 S[16][2];
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const float4 t = __ldcs(reinterpret_cast<const float4 *>(st + (size_t)(16 * warp + r) * D + 4 * lane));
    S[r][0] = make_float2(t.x, t.y);
    S[r][1] = make_float2(t.z, t.w);
  }
  // With two CTAs per SM the loads above leave HBM idle while the CTAs compute. Keep it busy
  // by asking for the state and the token rows of the CTA that starts about one wave later
  // (they are in L2 by the time that CTA loads them): bulk L2 prefetches, no registers held.
  if (warp < 2 && p.prefetch_dist > 0) {
    const long long nb = (long long)blockIdx.x + p.prefetch_dist;
    if (nb < (long long)gridDim.x) {
      const int nseq = (int)(nb / H), nh = (int)(nb % H);
      if (warp == 0 && lane < 4) {   // the state, four quarters of 16 KiB
        const int nslot = p.state_indices ? p.state_indices[nseq] : nseq;
        if (!p.state_indices || (nslot >= 0 && nslot < p.n_slots)) {
          const float *ns = p.state + ((size_t)nslot * H + nh) * D * D + (size_t)lane * (D * D / 4);
          prefetch_l2(ns, D * D * (int)sizeof(float) / 4);
        }
      } else if (warp == 1 && lane < 4 * LS) {   // one row of q, k, v or g per lane, all LS slots
        const int arr = lane / LS, l = lane % LS;
        const size_t row = ((size_t)nseq * LS + l) * H + nh;
        const int esz = arr == 3 ? (int)sizeof(float) : (int)sizeof(IO);
        const void *base = arr == 0 ? p.q : arr == 1 ? p.k : arr == 2 ? p.v : static_cast<const void *>(p.g);
        const char *src = static_cast<const char *>(base) + row * D * esz;
        prefetch_l2(src, D * esz);
      }
    }
  }

  cp_async_wait_all();
  __syncthreads();

  // L2 normalisation (one warp per token), v to fp32, and the running gate sums (one thread
  // per channel, on the last four warps: the first L warps normalise)
  if (warp < L) {
    float x[4], y[4], sq = 0.f, sk = 0.f, qk = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[j] = to_f(raw[(size_t)warp * D + lane + 32 * j]);
      y[j] = to_f(raw[(size_t)(L + warp) * D + lane + 32 * j]);
      sq = fmaf(x[j], x[j], sq);
      sk = fmaf(y[j], y[j], sk);
      qk = fmaf(x[j], y[j], qk);
    }
#pragma unroll
    for (int m = 16; m; m >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, m);
      sk += __shfl_xor_sync(0xffffffffu, sk, m);
      qk += __shfl_xor_sync(0xffffffffu, qk, m);
    }
    const float rq = p.scale * rsqrtf(sq + 1e-6f), rk = rsqrtf(sk + 1e-6f);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      sm.q[warp][lane + 32 * j] = x[j] * rq;
      sm.k[warp][lane + 32 * j] = y[j] * rk;
    }
    if (lane == 0) sm.b[warp][warp] = qk * rq * rk;
  }
  for (int idx = tid; idx < L * D; idx += STEP_THREADS) sm.v[idx / D][idx % D] = to_f(raw[(size_t)2 * L * D + idx]);
  if (tid >= STEP_THREADS - D) {
    const int c = tid - (STEP_THREADS - D);
    float run = 0.f;
    for (int l = 0; l < L; ++l) {
      run += sm.G[l][c];
      sm.G[l][c] = run;
    }
  }
  __syncthreads();

  // decayed vectors, and the token-token couplings a_lm, b_lm (m < l)
  for (int idx = tid; idx < L * D; idx += STEP_THREADS) {
    const int l = idx / D, c = idx % D;
    const float Gl = sm.G[l][c], kk = sm.k[l][c], gam = __expf(Gl);
    sm.kt[l][c] = gam * kk;
    sm.qt[l][c] = gam * sm.q[l][c];
    sm.kc[l][c] = A > 0 ? __expf(sm.G[A - 1][c] - Gl) * kk : 0.f;
  }
  if (tid < D) sm.gA[tid] = A > 0 ? __expf(sm.G[A - 1][tid]) : 1.f;
  for (int pr = warp; pr < L * (L - 1) / 2; pr += STEP_THREADS / 32) {
    int l = 1, m = pr;   // pair index -> (l, m) with m < l
    while (m >= l) {
      m -= l;
      ++l;
    }
    float sa = 0.f, sb = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = lane + 32 * j;
      const float e = __expf(sm.G[l][c] - sm.G[m][c]) * sm.k[m][c];
      sa = fmaf(e, sm.k[l][c], sa);
      sb = fmaf(e, sm.q[l][c], sb);
    }
#pragma unroll
    for (int s = 16; s; s >>= 1) {
      sa += __shfl_xor_sync(0xffffffffu, sa, s);
      sb += __shfl_xor_sync(0xffffffffu, sb, s);
    }
    if (lane == 0) {
      sm.a[l][m] = sa;
      sm.b[l][m] = sb;
    }
  }
  __syncthreads();

  // sweep 1: partial column sums of S0^T kt_l and S0^T qt_l over this warp's rows, two tokens at a time
  for (int l0 = 0; l0 < L; l0 += 2) {
    const bool two = l0 + 1 < L;
    const int l1 = two ? l0 + 1 : l0;
    float2 acc[4][2];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = make_float2(0.f, 0.f);
#pragma unroll
    for (int r4 = 0; r4 < 16; r4 += 4) {
      const int c = 16 * warp + r4;
      const float4 k0 = *reinterpret_cast<const float4 *>(&sm.kt[l0][c]);
      const float4 q0 = *reinterpret_cast<const float4 *>(&sm.qt[l0][c]);
      const float4 k1 = *reinterpret_cast<const float4 *>(&sm.kt[l1][c]);
      const float4 q1 = *reinterpret_cast<const float4 *>(&sm.qt[l1][c]);
      const float kv0[4] = {k0.x, k0.y, k0.z, k0.w}, qv0[4] = {q0.x, q0.y, q0.z, q0.w};
      const float kv1[4] = {k1.x, k1.y, k1.z, k1.w}, qv1[4] = {q1.x, q1.y, q1.z, q1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          acc[0][j] = __ffma2_rn(S[r4 + i][j], dup2(kv0[i]), acc[0][j]);
          acc[1][j] = __ffma2_rn(S[r4 + i][j], dup2(qv0[i]), acc[1][j]);
          acc[2][j] = __ffma2_rn(S[r4 + i][j], dup2(kv1[i]), acc[2][j]);
          acc[3][j] = __ffma2_rn(S[r4 + i][j], dup2(qv1[i]), acc[3][j]);
        }
      }
    }
    const int nv = two ? 4 : 2;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i < nv)
        *reinterpret_cast<float4 *>(&red[((size_t)warp * NV + 2 * l0 + i) * D + 4 * lane]) =
            make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
  }
  __syncthreads();

  // the token-token solve, one value column per thread: the 8 row-group partials of this column
  // summed in a fixed order, then the outputs of all L tokens
  if (tid < D) {
    IO *o = static_cast<IO *>(p.o);
    float u[STEP_MAX_L];
#pragma unroll
    for (int l = 0; l < STEP_MAX_L; ++l) {
      if (l < L) {
        float w = 0.f, ol = 0.f;
#pragma unroll
        for (int g8 = 0; g8 < 8; ++g8) {
          w += red[((size_t)g8 * NV + 2 * l) * D + tid];
          ol += red[((size_t)g8 * NV + 2 * l + 1) * D + tid];
        }
#pragma unroll
        for (int m = 0; m < l; ++m) {
          w = fmaf(sm.a[l][m], u[m], w);
          ol = fmaf(sm.b[l][m], u[m], ol);
        }
        u[l] = sm.beta[l] * (sm.v[l][tid] - w);
        ol = fmaf(sm.b[l][l], u[l], ol);
        sm.U[l][tid] = u[l];
        o[(((size_t)seq * LS + F + l) * H + h) * D + tid] = from_f<IO>(ol);
      }
    }
  }
  __syncthreads();

  // sweep 2: S_A = Diag(gamma_A) S0 + sum_{m<A} kc_m u_m^T, then the one write-back
  if (A > 0) {
#pragma unroll
    for (int r4 = 0; r4 < 16; r4 += 4) {
      const float4 g4 = *reinterpret_cast<const float4 *>(&sm.gA[16 * warp + r4]);
      const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        S[r4 + i][0] = __fmul2_rn(S[r4 + i][0], dup2(gv[i]));
        S[r4 + i][1] = __fmul2_rn(S[r4 + i][1], dup2(gv[i]));
      }
    }
    for (int m = 0; m < A; ++m) {
      const float4 u4 = *reinterpret_cast<const float4 *>(&sm.U[m][4 * lane]);
      const float2 u0 = make_float2(u4.x, u4.y), u1 = make_float2(u4.z, u4.w);
#pragma unroll
      for (int r4 = 0; r4 < 16; r4 += 4) {
        const float4 c4 = *reinterpret_cast<const float4 *>(&sm.kc[m][16 * warp + r4]);
        const float cv[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          S[r4 + i][0] = __ffma2_rn(dup2(cv[i]), u0, S[r4 + i][0]);
          S[r4 + i][1] = __ffma2_rn(dup2(cv[i]), u1, S[r4 + i][1]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 16; ++r)
      __stcs(reinterpret_cast<float4 *>(st + (size_t)(16 * warp + r) * D + 4 * lane),
             make_float4(S[r][0].x, S[r][0].y, S[r][1].x, S[r][1].y));
  }
}

template <typename IO, bool PAD>
static cudaError_t launch_step_t(const StepParams &p, unsigned grid, cudaStream_t s) {
  // Dynamic shared memory: 8 row-group partials, 2L vectors each.
  constexpr int max_smem = 8 * 2 * STEP_MAX_L * D * (int)sizeof(float);
  const int smem = 8 * 2 * p.steps * D * (int)sizeof(float);
  // static + dynamic exceeds the 48 KiB default: opt in (per device, idempotent)
  const cudaError_t e =
      cudaFuncSetAttribute(kda_step_kernel<IO, PAD>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  // prefetch distance: the CTAs resident at once (one wave)
  int dev = 0, sms = 0, per_sm = 0;
  StepParams q = p;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_step_kernel<IO, PAD>, STEP_THREADS, smem) ==
          cudaSuccess)
    q.prefetch_dist = sms * per_sm;
  else
    q.prefetch_dist = 0;
  kda_step_kernel<IO, PAD><<<grid, STEP_THREADS, smem, s>>>(q);
  return cudaGetLastError();
}

cudaError_t launch_step(const StepParams &p, bool f32, cudaStream_t s) {
  const unsigned grid = (unsigned)((long long)p.n_seqs * p.heads);
  if (grid == 0) return cudaSuccess;
  const bool pad = p.first_slot != nullptr;
  if (f32) return pad ? launch_step_t<float, true>(p, grid, s) : launch_step_t<float, false>(p, grid, s);
  return pad ? launch_step_t<bf16, true>(p, grid, s) : launch_step_t<bf16, false>(p, grid, s);
}

}  // namespace kda
