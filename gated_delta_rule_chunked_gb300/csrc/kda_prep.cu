// kda_prep.cu -- chunk table and the chunk-parallel intra-chunk kernel of the fp32-I/O forward
// (the bf16 forward's intra-chunk kernel runs on tcgen05: kda_prep_tc.cu).
//
// For every (64-token chunk, head), independently of all other chunks:
//   1. Q/K L2 normalisation (the benchmark caption of the first page counts
//      "Q/K normalization and gate scan" as part of the KDA core);
//   2. the gate scan G_r = sum_{i<=r} g_i per key channel, restarted per chunk
//      (kept in log2 units);
//   3. the gated Gram blocks A_rj = sum_c k^_rc k^_jc exp(G_rc-G_jc) (j<r) and
//      B_rj = sum_c q^_rc k^_jc exp(G_rc-G_jc) (j<=r) in exact fp32 products (the fp32
//      I/O tolerance leaves no room for TF32 operands);
//   4. the WY/UT transform T = (I + Diag(beta) A)^-1 (16x16 diagonal blocks by
//      forward substitution, off-diagonal blocks by fp32 block products);
//   5. the operands the sequential state scan needs, written as one record, and, for the
//      backward, A (strict lower, without beta) and T in plain fp32 [64][64] arrays.
//
// Gating factorisation. exp(G_r - G_j) is split into two bounded factors so the
// Gram products run as plain matrix multiplies. With 16-token sub-blocks and
// E_a = G at the last row of sub-block a (E_-1 = 0), for r in sub-block a and j
// in sub-block b <= a:
//   exp(G_r - G_j) = exp(G_r - E_{a-1}) * exp(E_b - G_j) * exp(E_{a-1} - E_b)
// The first two factors are <= 1 (one per row, stored once), the third is a
// per-channel vector per sub-block pair: <= 1 for b < a and, for b = a,
// exp(-(sum of g over the sub-block)), which the library's precondition
// (16-token gate sums >= -80) keeps finite. Within a sub-block the local running
// sum of g gives G_r - E_{a-1} directly, so no large G is ever subtracted.
// This is this library's kernel design, not taken from the pages.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc05.cuh"

namespace kda {

// ------------------------------------------------------------ chunk table
__global__ void chunk_table_kernel(const int *cu_in, int n_seqs, long long total, int *cu_out,
                                   int *chunk_off) {
  // single block: cu_out = cu_in (or equal lengths), chunk_off = prefix sum of ceil(L/64)
  __shared__ int carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const long long per = n_seqs ? total / n_seqs : 0;
  for (int base = 0; base < n_seqs; base += blockDim.x) {
    const int i = base + threadIdx.x;
    int nch = 0;
    if (i < n_seqs) {
      const long long s0 = cu_in ? cu_in[i] : per * i;
      const long long s1 = cu_in ? cu_in[i + 1] : per * (i + 1);
      cu_out[i] = (int)s0;
      if (i == n_seqs - 1) cu_out[n_seqs] = (int)s1;
      const long long len = s1 > s0 ? s1 - s0 : 0;
      nch = (int)((len + CH - 1) / CH);
    }
    // block-wide inclusive scan of nch (Hillis-Steele in shared memory)
    __shared__ int buf[1024];
    buf[threadIdx.x] = nch;
    __syncthreads();
    for (int o = 1; o < (int)blockDim.x; o <<= 1) {
      const int add = threadIdx.x >= (unsigned)o ? buf[threadIdx.x - o] : 0;
      __syncthreads();
      buf[threadIdx.x] += add;
      __syncthreads();
    }
    if (i < n_seqs) chunk_off[i] = carry + buf[threadIdx.x] - nch;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry += buf[threadIdx.x];
    __syncthreads();
  }
  if (threadIdx.x == 0) chunk_off[n_seqs] = carry;
}

cudaError_t launch_chunk_table(const int *cu_in, int n_seqs, long long total, int *cu_out, int *chunk_off,
                               cudaStream_t s) {
  chunk_table_kernel<<<1, 1024, 0, s>>>(cu_in, n_seqs, total, cu_out, chunk_off);
  return cudaGetLastError();
}

// ------------------------------------------------------------ the prep kernel
constexpr int PREP_THREADS = 256;
constexpr int LDF = 136;   // padded fp32 row of the 64x128 factor tiles: 136 = 8 (mod 32) makes the
                           // 8-byte fragment reads of the Gram products and the Kt reads of W conflict-free
constexpr int LDS64 = 68;  // padded fp32 row of 64x64 tiles
constexpr int LDP = 24;    // padded fp32 row of the 16x16 solver scratch

struct PrepSmem2 {
  static constexpr int TILE = 64 * LDF * 4;
  static constexpr int KL = 0, QL = TILE, R = 2 * TILE;     // fp32 [64][LDF] each
  static constexpr int DV = 3 * TILE;                        // fp32 [10][128] pair factors
  static constexpr int TOT = DV + 10 * 512;                  // fp32 [4][128] sub-block gate sums
  static constexpr int RQ = TOT + 4 * 512, RK = RQ + 256, BETA = RK + 256;
  static constexpr int BAR = BETA + 256;                     // mbarrier of the staging copies
  static constexpr int BYTES = BAR + 16;
  // after the Gram products QL and R are dead
  static constexpr int LM = QL;                              // fp32 [64][LDS64]  Diag(beta) A
  static constexpr int TT = LM + 64 * LDS64 * 4;             // fp32 [64][LDS64]  T, then T Diag(beta)
  static constexpr int SCR = TT + 64 * LDS64 * 4;            // fp32 4 x [16][LDP]
  static_assert(SCR + 4 * 16 * LDP * 4 <= DV, "solver tiles overlap the vectors");
};

__device__ __forceinline__ void zero4(float (&a)[4]) { a[0] = a[1] = a[2] = a[3] = 0.f; }

__device__ __forceinline__ void pair_of(int p, int &a, int &b) {
  a = p >= 6 ? 3 : (p >= 3 ? 2 : (p >= 1 ? 1 : 0));
  b = p - a * (a + 1) / 2;
}

// Gram units. Unit u = (pair, n-tile): rows 16 pa.. of KL and of QL against the 8 columns
// 16 pb + 8 nt.. of R scaled by the pair factors D_{pa,pb}:
//   ak += KL_pa diag(d) R_cols^T (the A side),  aq += QL_pa diag(d) R_cols^T (the B side),
// both 16 x 8 in the m16n8 accumulator layout. The two products share the scaled R
// fragments. In the TF32 form the contraction order inside each group of 8 channels is
// permuted (fragment k = q reads channel 2q, k = q + 4 reads 2q + 1), so every fragment pair
// is one 8-byte shared-memory read; KL and QL hold values already rounded to TF32. NU units
// per warp run interleaved (independent accumulator chains).
struct GramUnit {
  const float *kl, *ql, *rr, *d;   // KL, QL rows of the row block; R rows of the n-tile; pair factors
};
template <int NU>
__device__ __forceinline__ void gram_units(float (&ak)[3][4], float (&aq)[3][4], const GramUnit (&u)[3]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int v = 0; v < NU; ++v)
    for (int c = 0; c < 128; ++c) {
      const float d = u[v].d[c];
      const float k0 = u[v].kl[g * LDF + c], k1 = u[v].kl[(g + 8) * LDF + c];
      const float q0 = u[v].ql[g * LDF + c], q1 = u[v].ql[(g + 8) * LDF + c];
      const float r0 = u[v].rr[(2 * q) * LDF + c] * d, r1 = u[v].rr[(2 * q + 1) * LDF + c] * d;
      ak[v][0] = fmaf(k0, r0, ak[v][0]);
      ak[v][1] = fmaf(k0, r1, ak[v][1]);
      ak[v][2] = fmaf(k1, r0, ak[v][2]);
      ak[v][3] = fmaf(k1, r1, ak[v][3]);
      aq[v][0] = fmaf(q0, r0, aq[v][0]);
      aq[v][1] = fmaf(q0, r1, aq[v][1]);
      aq[v][2] = fmaf(q1, r0, aq[v][2]);
      aq[v][3] = fmaf(q1, r1, aq[v][3]);
    }
}

// acc (16x16) += A[16][16] * B[16][16], row-major fp32 with leading dims lda, ldb, in the m16n8
// accumulator layout (exact fp32 FMAs).
__device__ __forceinline__ void mm16(float (&acc)[2][4], const float *A, int lda, const float *B, int ldb) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
#pragma unroll 4
  for (int k = 0; k < 16; ++k) {
    const float a0 = A[g * lda + k], a1 = A[(g + 8) * lda + k];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float b0 = B[k * ldb + 8 * nt + 2 * q], b1 = B[k * ldb + 8 * nt + 2 * q + 1];
      acc[nt][0] = fmaf(a0, b0, acc[nt][0]);
      acc[nt][1] = fmaf(a0, b1, acc[nt][1]);
      acc[nt][2] = fmaf(a1, b0, acc[nt][2]);
      acc[nt][3] = fmaf(a1, b1, acc[nt][3]);
    }
  }
}

__global__ void __launch_bounds__(PREP_THREADS, 2) kda_prep_kernel(const __grid_constant__ PrepParams p) {
  using S = PrepSmem2;
  typedef float E;
  extern __shared__ __align__(128) char smem[];
  // head-fastest block order: the CTAs resident at one time cover whole token rows
  // [t][all heads][d] and consecutive chunk records (DRAM pages read whole), not one head's
  // rows strided by heads x d
  const int H = p.geo.heads, h = (int)(blockIdx.x % (unsigned)H), chunk = (int)(blockIdx.x / (unsigned)H);
  ChunkRef ref;
  if (!chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, chunk, ref)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
  float *rq = (float *)(smem + S::RQ), *rk = (float *)(smem + S::RK), *sb = (float *)(smem + S::BETA);
  float *KL = (float *)(smem + S::KL), *QL = (float *)(smem + S::QL), *RR = (float *)(smem + S::R);
  float(*dv)[128] = (float(*)[128])(smem + S::DV);
  float(*tot)[128] = (float(*)[128])(smem + S::TOT);
  const ImgLayout L(sizeof(E));
  const size_t rid = (size_t)chunk * H + h;
  char *trec = (char *)p.img + rid * L.bytes;   // the tile record the fp32 scan reads
  // the backward's copy of A (strict lower, without beta) and T, plain [64][64] fp32 each
  float *aux = p.aux ? p.aux + rid * 2 * 64 * 64 : nullptr;

  // 0. stage the chunk's q, k (io type) and g (fp32) in shared memory with three TMA boxes:
  //    q in the KL tile, k in the R tile (plain rows), g in the QL tile (dense 128-float rows);
  //    rows past the sequence end are zeroed. All three tiles are rewritten only after their
  //    contents have been consumed.
  constexpr int QROW = D * (int)sizeof(E);            // bytes of one staged q / k row
  const E *sq_ = (const E *)KL, *sk_ = (const E *)RR;
  {
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::BAR);
    if (tid == 0) {
      mbar_init(bar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      const int t0i = (int)ref.t0;
      mbar_expect_tx(bar, 2 * CH * QROW + CH * D * 4);
      tc::tma_load_3d(KL, &p.tm_q, 0, h, t0i, bar);
      tc::tma_load_3d(RR, &p.tm_k, 0, h, t0i, bar);
      tc::tma_load_3d(QL, &p.tm_g, 0, h, t0i, bar);
    }
    if (tid < 64) sb[tid] = tid < ref.len ? p.beta[(size_t)(ref.t0 + tid) * H + h] : 0.f;
    const bool ok = mbar_wait(bar, 0);
    if (ok && ref.len < CH) {   // the boxes hold the next sequence's rows there
      for (int idx = tid; idx < (CH - ref.len) * (QROW / 16); idx += PREP_THREADS) {
        const int r = ref.len + idx / (QROW / 16), ch = idx % (QROW / 16);
        *reinterpret_cast<uint4 *>((char *)KL + r * QROW + 16 * ch) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>((char *)RR + r * QROW + 16 * ch) = make_uint4(0u, 0u, 0u, 0u);
      }
      for (int idx = tid; idx < (CH - ref.len) * (D / 4); idx += PREP_THREADS) {
        const int r = ref.len + idx / (D / 4), ch = idx % (D / 4);
        *reinterpret_cast<float4 *>(QL + r * D + 4 * ch) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (!__syncthreads_and(ok)) {
      report(p.status, ERR_TIMEOUT);
      return;
    }
  }
  // 1. row norms: 4 threads per row, 32 channels each
  {
    const int r = tid >> 2, part = tid & 3;
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      const float2 a = ld2(sq_ + r * D + part * 32 + c), b = ld2(sk_ + r * D + part * 32 + c);
      sq = fmaf(a.x, a.x, fmaf(a.y, a.y, sq));
      sk = fmaf(b.x, b.x, fmaf(b.y, b.y, sk));
    }
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 2);
    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
    sk += __shfl_xor_sync(0xffffffffu, sk, 2);
    if (part == 0) {
      rq[r] = p.scale * rsqrtf(sq + 1e-6f);
      rk[r] = rsqrtf(sk + 1e-6f);
    }
  }
  // 2. gate scan and factors: thread = (channel pair cp, sub-block a)
  const int cp = tid & 63, a = tid >> 6, c0 = 2 * cp;
  float2 cs[SUB];
  float2 qpair[SUB], kpair[SUB];   // this thread's raw q, k (rows a*SUB.., channels c0, c0+1)
  {
#pragma unroll
    for (int i = 0; i < SUB; ++i) {
      const int r = a * SUB + i;
      cs[i] = *reinterpret_cast<const float2 *>(QL + r * D + c0);
      qpair[i] = ld2(sq_ + r * D + c0);
      kpair[i] = ld2(sk_ + r * D + c0);
    }
    float2 run = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < SUB; ++i) {
      run.x = fmaf(cs[i].x, LOG2E, run.x);
      run.y = fmaf(cs[i].y, LOG2E, run.y);
      cs[i] = run;                          // G_r - E_{a-1}, log2 units
    }
    tot[a][c0] = run.x;
    tot[a][c0 + 1] = run.y;
  }
  __syncthreads();
  {
    // E_{a-1}, E_a, E_3 per channel (running sums of the sub-block totals)
    float em[2] = {0.f, 0.f}, ea[2], e3[2] = {0.f, 0.f}, eb[2] = {0.f, 0.f};
#pragma unroll
    for (int b = 0; b < NSUB; ++b) {
      const float t0 = tot[b][c0], t1 = tot[b][c0 + 1];
      if (b < a) { em[0] += t0; em[1] += t1; }
      e3[0] += t0;
      e3[1] += t1;
    }
    ea[0] = em[0] + tot[a][c0];
    ea[1] = em[1] + tot[a][c0 + 1];
    // pair factors D_{a,b} = 2^(E_{a-1} - E_b), b <= a
#pragma unroll
    for (int b = 0; b < NSUB; ++b) {
      eb[0] += tot[b][c0];
      eb[1] += tot[b][c0 + 1];
      if (b <= a) {
        const int pr = a * (a + 1) / 2 + b;
        dv[pr][c0] = exp2f(em[0] - eb[0]);
        dv[pr][c0 + 1] = exp2f(em[1] - eb[1]);
      }
    }
    const float pa0 = exp2f(em[0]), pa1 = exp2f(em[1]);                       // exp(E_{a-1})
    const float fa0 = exp2f(e3[0] - ea[0]), fa1 = exp2f(e3[1] - ea[1]);       // exp(E_3 - E_a)
    const float ta0 = tot[a][c0], ta1 = tot[a][c0 + 1];                       // E_a - E_{a-1}
    Tile<E, 128> tqt((E *)(trec + L.qt)), tkt((E *)(trec + L.kt)), tkh((E *)(trec + L.kh));
    float kh0v[SUB], kh1v[SUB];
#pragma unroll
    for (int i = 0; i < SUB; ++i) {
      const int r = a * SUB + i;
      const float2 qv = qpair[i], kv = kpair[i];
      const float x0 = exp2f(cs[i].x), x1 = exp2f(cs[i].y);
      const float y0 = exp2f(ta0 - cs[i].x), y1 = exp2f(ta1 - cs[i].y);
      const float qh0 = qv.x * rq[r], qh1 = qv.y * rq[r], kh0 = kv.x * rk[r], kh1 = kv.y * rk[r];
      const float kl0 = kh0 * x0, kl1 = kh1 * x1, ql0 = qh0 * x0, ql1 = qh1 * x1;
      const float rr0 = kh0 * y0, rr1 = kh1 * y1;
      *reinterpret_cast<float2 *>(KL + r * LDF + c0) = make_float2(kl0, kl1);
      *reinterpret_cast<float2 *>(QL + r * LDF + c0) = make_float2(ql0, ql1);
      *reinterpret_cast<float2 *>(RR + r * LDF + c0) = make_float2(rr0, rr1);
      kh0v[i] = rr0 * fa0;                        // Kh = k^ exp(G_last - G_r)
      kh1v[i] = rr1 * fa1;
      st2(tqt.at(r, c0), ql0 * pa0, ql1 * pa1);                 // Qt = q^ exp(G_r)
      st2(tkt.at(r, c0), kl0 * pa0, kl1 * pa1);                 // Kt = k^ exp(G_r)
      st2(tkh.at(r, c0), kh0v[i], kh1v[i]);
    }
    if (a == 0) *reinterpret_cast<float2 *>(trec + L.gc + c0 * 4) = make_float2(exp2f(e3[0]), exp2f(e3[1]));
  }
  __syncthreads();
  // 3. Gram products: 20 units (pair, n-tile), warp w takes units w, w + 8, w + 16
  float acc[3][4], accq[3][4];
  {
    GramUnit un[3];
#pragma unroll
    for (int v = 0; v < 3; ++v) {
      zero4(acc[v]);
      zero4(accq[v]);
      const int unit = min(warp + 8 * v, 19), pr = unit >> 1;
      int pa, pb;
      pair_of(pr, pa, pb);
      un[v].kl = KL + pa * SUB * LDF;
      un[v].ql = QL + pa * SUB * LDF;
      un[v].rr = RR + (pb * SUB + 8 * (unit & 1)) * LDF;
      un[v].d = dv[pr];
    }
    if (warp < 4) gram_units<3>(acc, accq, un);
    else gram_units<2>(acc, accq, un);
  }
  __syncthreads();   // QL and R are free from here on
  {
    float *Lm = (float *)(smem + S::LM);
    Tile<E, 64> bm((E *)(trec + L.bm));
#pragma unroll
    for (int v = 0; v < 3; ++v) {
      const int unit = warp + 8 * v;
      if (unit >= 20) continue;
      int pa, pb;
      pair_of(unit >> 1, pa, pb);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = pa * SUB + g + 8 * hh, j = pb * SUB + 8 * (unit & 1) + 2 * q;
        const float v0 = accq[v][2 * hh], v1 = accq[v][2 * hh + 1];
        const float b0 = j <= r ? v0 : 0.f, b1 = j + 1 <= r ? v1 : 0.f;
        st2(bm.at(r, j), b0, b1);
        const float w0 = acc[v][2 * hh], w1 = acc[v][2 * hh + 1];
        const float a0 = j < r ? w0 : 0.f, a1 = j + 1 < r ? w1 : 0.f;
        *reinterpret_cast<float2 *>(Lm + r * LDS64 + j) = make_float2(sb[r] * a0, sb[r] * a1);
        if (aux) *reinterpret_cast<float2 *>(aux + r * 64 + j) = make_float2(a0, a1);
      }
    }
    // zero the sub-blocks of Bm (and of A for the backward) above the diagonal
    for (int idx = tid; idx < 64 * 32; idx += PREP_THREADS) {
      const int r = idx >> 5, j = (idx & 31) * 2;
      if ((j >> 4) > (r >> 4)) {
        st2(bm.at(r, j), 0.f, 0.f);
        if (aux) *reinterpret_cast<float2 *>(aux + r * 64 + j) = make_float2(0.f, 0.f);
      }
    }
  }
  __syncthreads();
  // 4. T = (I + Lm)^-1: diagonal sub-blocks by forward substitution (warps 0..3), then the
  //    off-diagonal blocks level by level on warps 0..3; then Tb = T Diag(beta) into the record
  //    (and T for the backward).
  {
    const float *Lm = (const float *)(smem + S::LM);
    float *T = (float *)(smem + S::TT);
    if (warp < NSUB) {
      const int ab = warp, j = lane & 15;
      float x[SUB];
#pragma unroll
      for (int i = 0; i < SUB; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
      for (int i = 1; i < SUB; ++i) {
        float s_ = 0.f;
#pragma unroll
        for (int m = 0; m < i; ++m) s_ = fmaf(Lm[(ab * SUB + i) * LDS64 + ab * SUB + m], x[m], s_);
        if (i > j) x[i] = -s_;
      }
      if (lane < SUB) {
#pragma unroll
        for (int i = 0; i < SUB; ++i) T[(ab * SUB + i) * LDS64 + ab * SUB + j] = x[i];
      }
    } else {
      // warps 4..7 zero the blocks above the diagonal
      for (int idx = tid - 128; idx < 64 * 64; idx += 128) {
        const int r = idx >> 6, j = idx & 63;
        if ((j >> 4) > (r >> 4)) T[r * LDS64 + j] = 0.f;
      }
    }
    __syncthreads();
    // off-diagonal sub-blocks by levels: T_ab = -T_aa * sum_{m=b}^{a-1} Lm_am T_mb
    float *P = (float *)(smem + S::SCR) + warp * 16 * LDP;
    for (int d = 1; d < NSUB; ++d) {
      const int b = warp, ab = warp + d;
      if (warp < NSUB && ab < NSUB) {
        float pacc[2][4];
        zero(pacc);
        for (int m = b; m < ab; ++m)
          mm16(pacc, Lm + ab * SUB * LDS64 + m * SUB, LDS64, T + m * SUB * LDS64 + b * SUB, LDS64);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          *reinterpret_cast<float2 *>(P + g * LDP + 8 * nt + 2 * q) = make_float2(pacc[nt][0], pacc[nt][1]);
          *reinterpret_cast<float2 *>(P + (g + 8) * LDP + 8 * nt + 2 * q) = make_float2(pacc[nt][2], pacc[nt][3]);
        }
        __syncwarp();
        float tacc[2][4];
        zero(tacc);
        mm16(tacc, T + ab * SUB * LDS64 + ab * SUB, LDS64, P, LDP);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          float *dst = T + (ab * SUB + g) * LDS64 + b * SUB + 8 * nt + 2 * q;
          *reinterpret_cast<float2 *>(dst) = make_float2(-tacc[nt][0], -tacc[nt][1]);
          *reinterpret_cast<float2 *>(dst + 8 * LDS64) = make_float2(-tacc[nt][2], -tacc[nt][3]);
        }
        __syncwarp();
      }
      __syncthreads();
    }
    Tile<E, 64> tb((E *)(trec + L.tb));
    for (int idx = tid; idx < 64 * 32; idx += PREP_THREADS) {
      const int r = idx >> 5, j = (idx & 31) * 2;
      const float t0v = T[r * LDS64 + j], t1v = T[r * LDS64 + j + 1];
      st2(tb.at(r, j), t0v * sb[j], t1v * sb[j + 1]);
      if (aux) *reinterpret_cast<float2 *>(aux + 64 * 64 + r * 64 + j) = make_float2(t0v, t1v);
    }
  }
}

cudaError_t launch_prep(const PrepParams &p, bool f32, cudaStream_t s) {
  if (p.geo.max_chunks == 0) return cudaSuccess;
  if (!f32) return cudaErrorInvalidValue;   // the bf16 forward runs launch_prep_tc
  using S = PrepSmem2;
  cudaError_t e = cudaFuncSetAttribute(kda_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::BYTES);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.geo.max_chunks * p.geo.heads;   // head-fastest: see the kernel
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kda_prep_kernel<<<(unsigned)blocks, PREP_THREADS, S::BYTES, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
