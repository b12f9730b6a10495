// kda_prep_tc.cu -- the intra-chunk kernel of the bf16 forward on 5th-generation tensor cores.
//
// For every (64-token chunk, head), independently of all other chunks (the KDA
// paragraph of "Kimi K3 on Fireworks: Fast RL at frontier scale": chunk-local work in
// parallel, a compact state between chunks):
//   1. Q/K L2 normalisation and the per-channel gate scan (the benchmark caption of
//      "KDA：从循环记忆到高效 GPU 执行" counts both as part of the KDA core);
//   2. the gated Gram blocks A_rj = sum_c k^_rc k^_jc e^{G_rc - G_jc} (j < r) and
//      B_rj = sum_c q^_rc k^_jc e^{G_rc - G_jc} (j <= r) as tcgen05 kind::tf32 products
//      accumulated in tensor memory;
//   3. the WY/UT transform T = (I + Diag(beta) A)^-1: the four 16 x 16 diagonal blocks by
//      forward substitution, the rest as a short series of tcgen05 products;
//   4. W = T Diag(beta) Kt as one more tcgen05 product, and the record the scans read.
//
// Gating. e^{G_r - G_j} is split at one reference per 16-row block a of r: with E_a the
// gate sum at the end of sub-block a (E_-1 = 0),
//   e^{G_r - G_j} = e^{G_r - E_{a-1}} * e^{E_{a-1} - G_j}.
// The left factor is <= 1 (one per row: KL = k^ e^{G - E_{a-1}}, QL likewise). The right
// factor RA^(a)_j = k^_j e^{E_{a-1} - G_j} is <= 1 for j before block a and at most
// e^{80} inside it under the library's precondition (16-token gate sums >= -80), so every
// tf32 operand stays in range. The right factors of the four row blocks (16, 32, 48 and 64
// rows j) are stacked into the B operand (N = 160) of one product against the A operand
// [KL; QL] (M = 128): D[m][n] = A_rj (m = r) or B_rj (m = 64 + r) for the stacked column
// n = (block of r, j), so each thread reads its own row of A or B out of tensor memory.
// The contraction over the 128 key channels runs in two halves of 64 so the operands fit
// beside a second CTA on the SM.
//
// UT transform. With Lm = Diag(beta) A, D = the inverse of its block diagonal (four 16 x 16
// forward substitutions) and N its strictly block-lower part, I + Lm = D^-1 (I + D N), so
// T = (I + D N)^-1 D = (I + E')(I + E'^2) D with E' = -D N (E' is strictly block lower over
// four blocks, so its fourth power vanishes and the product is exact). Three rounds of
// tcgen05 products give E', then E' D and E'^2 together, then E'^2 (D + E' D); they run in
// the transposed orientation where that lets each read-out of tensor memory write the next
// operand row by row.
// This is this library's design, not taken from the pages.
//
// Every wait is bounded; on a timeout the CTA reports KDA_ERR_TIMEOUT, frees its tensor
// memory and returns.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc05.cuh"

namespace kda {
namespace {

constexpr int PT_THREADS = 256;

struct PtSmem {
  // staging: q, k bf16 [64][128] plain rows, g fp32 [64][128] (three TMA boxes)
  static constexpr int STQ = 0, STK = 16384, STG = 32768;
  // local gate sums G_r - E_{a-1} (log2 units), fp32 [64][128] plain rows, over the q, k staging
  static constexpr int CS = 0;
  // Gram operands of one channel half: tf32 tiles, K-major, 128-byte swizzle, two K-blocks of 32 channels
  static constexpr int GA = 32768;    // [2][128][128 B]  [KL; QL]                  (A, M = 128)
  static constexpr int GB = 65536;    // [2][160][128 B]  stacked right factors     (B, N = 160)
  // after the Gram, over the dead operands
  static constexpr int NT = 0;        // -N^T [j][m]; then F^T = (D + E' D)^T [j][m]
  static constexpr int DD = 16384;    // D [r][m]; then E'^T [j][m]; then E'^2 [r][m]
  static constexpr int DT = 32768;    // D^T [j][m]
  static constexpr int EP = 49152;    // E' [r][m]; then T [r][j] (W's A operand)
  static constexpr int BKT = 65536;   // (Diag(beta) Kt)^T [128 ch][64 tok], 2 K-blocks of 16 KB (W's B operand)
  static constexpr int LD = 98304;    // diagonal blocks of Lm: [4][16][17] fp32
  static constexpr int TOT = 98304;   // [4][128] sub-block gate sums (log2 units): phase 1 only, inside GB
  // live from phase 1 to the end, above GB
  static constexpr int RQ = GB + 2 * 160 * 128, RK = RQ + 256, SB = RK + 256;
  static constexpr int PA = SB + 256;           // [4][128] e^{E_{a-1}}
  static constexpr int PF = PA + 2048;          // [6][128] e^{E_{a'-1} - E_{a-1}}, pairs a < a'
  static constexpr int BAR = PF + 3072;         // [0] staging copies, [1] MMA commits, [2..3] Gram K-block buffers
  static constexpr int TSLOT = BAR + 32;
  static constexpr int BYTES = TSLOT + 16 + 1024;   // + alignment slack
};
static_assert(PtSmem::BYTES <= 115200, "two CTAs per SM");

constexpr uint32_t TCOLS = 256;    // tensor memory: Gram [0,160); UT products [0,64); W [128,256)
// first stacked column of row block a (which has 16 (a + 1) columns): 0, 16, 48, 96
__host__ __device__ constexpr int stack_off(int a) { return 8 * a * (a + 1); }
// index of the row-block pair a < a' in the factor table: (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
__host__ __device__ constexpr int pair_idx(int a, int ap) { return a * (7 - a) / 2 + (ap - a - 1); }

__device__ __forceinline__ float rtf32(float x) { return __uint_as_float(tf32(x)); }
// 2^x by the hardware approximation (relative error about 2^-22), results below 2^-126 flushed to
// zero: every gating factor here multiplies O(1) values, so such results are negligible
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// byte offset of fp32 element (row, k) of a K-major SW128 tile with `rows` rows
__device__ __forceinline__ uint32_t o32(int rows, int row, int k) { return tc::sw128_off32(rows, row, k); }


// Warp-collective: 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
  float x[16], y[16];
  tc::ld16(taddr, x);
  tc::ld16(taddr + 16, y);
  tc::wait_ld();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = x[i];
    v[16 + i] = y[i];
  }
}

// tf32 product of two 64-row K-major tiles over K = 64: D[tmem] = A B^T (M = 64, N = nrows_b)
__device__ __forceinline__ void mma64(uint32_t d, uint32_t sa, uint32_t sb, int nb, uint32_t b_kstride) {
  const uint32_t idesc = tc::idesc_tf32(64, nb);
#pragma unroll
  for (int kb = 0; kb < 2; ++kb)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      tc::mma_tf32(d, tc::desc_sw128(sa + 8192u * kb + 32u * ks), tc::desc_sw128(sb + b_kstride * kb + 32u * ks),
                   idesc, (kb | ks) != 0);
}

}  // namespace

__global__ void __launch_bounds__(PT_THREADS, 2) kda_prep_tc_kernel(const __grid_constant__ PrepParams p) {
  using S = PtSmem;
  extern __shared__ __align__(1024) char smem_raw[];
  char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // head-fastest block order: the CTAs resident together read whole token rows
  const int H = p.geo.heads, h = (int)(blockIdx.x % (unsigned)H), chunk = (int)(blockIdx.x / (unsigned)H);
  ChunkRef ref;
  if (!chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, chunk, ref)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool bwdrec = (p.tc_layout & 2) != 0;   // training forward: Kt, A and T for the backward
  const size_t rid = (size_t)chunk * H + h;
  char *rec = (char *)p.img + rid * TcRec::BYTES;
  char *ktrec = bwdrec ? (char *)p.img2 + rid * KtRec::BYTES : nullptr;
  float *auxA = bwdrec && p.aux ? p.aux + rid * (2 * 64 * 64) : nullptr;
  float *auxT = auxA ? auxA + 64 * 64 : nullptr;
  float *rq = (float *)(smem + S::RQ), *rk = (float *)(smem + S::RK), *sb = (float *)(smem + S::SB);
  float(*tot)[128] = (float(*)[128])(smem + S::TOT);
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::BAR);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + S::TSLOT);

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, TCOLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);   // this warp's lane quarter
  uint32_t mma_phase = 0;
  auto fail = [&]() {
    report(p.status, ERR_TIMEOUT);
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::dealloc(tmem, TCOLS);
  };
  // one commit of every MMA issued so far, then all threads wait for it
  auto mma_done = [&]() -> bool {
    const bool ok = mbar_wait(&bar[1], mma_phase);
    mma_phase ^= 1u;
    tc::fence_after();
    return __syncthreads_and(ok);
  };

  // ---------------------------------------------------------------- 0. staging
  {
    if (tid == 0) {
      const int t0i = (int)ref.t0;
      mbar_expect_tx(&bar[0], 2 * 16384 + 32768);
      tc::tma_load_3d(smem + S::STQ, &p.tm_q, 0, h, t0i, &bar[0]);
      tc::tma_load_3d(smem + S::STK, &p.tm_k, 0, h, t0i, &bar[0]);
      tc::tma_load_3d(smem + S::STG, &p.tm_g, 0, h, t0i, &bar[0]);
    }
    if (tid < 64) sb[tid] = tid < ref.len ? p.beta[(size_t)(ref.t0 + tid) * H + h] : 0.f;
    if (warp == 2 && p.prefetch_dist > 0) {
      // the staging boxes and betas of the CTA that starts about one wave later, into L2
      const long long nbk = (long long)blockIdx.x + p.prefetch_dist;
      ChunkRef nref;
      if (nbk < (long long)gridDim.x &&
          chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, (int)(nbk / H), nref)) {
        const int nh = (int)(nbk % H);
        if (lane == 0) tc::tma_prefetch_3d(&p.tm_q, 0, nh, (int)nref.t0);
        if (lane == 1) tc::tma_prefetch_3d(&p.tm_k, 0, nh, (int)nref.t0);
        if (lane == 2) tc::tma_prefetch_3d(&p.tm_g, 0, nh, (int)nref.t0);
      }
    }
    const bool ok = mbar_wait(&bar[0], 0);
    if (ok && ref.len < CH) {   // the boxes hold the next sequence's rows there
      for (int idx = tid; idx < (CH - ref.len) * 16; idx += PT_THREADS) {
        const int r = ref.len + (idx >> 4), c = idx & 15;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(smem + S::STQ + r * 256 + 16 * c) = z;
        *reinterpret_cast<uint4 *>(smem + S::STK + r * 256 + 16 * c) = z;
        *reinterpret_cast<uint4 *>(smem + S::STG + r * 512 + 32 * c) = z;
        *reinterpret_cast<uint4 *>(smem + S::STG + r * 512 + 32 * c + 16) = z;
      }
    }
    if (!__syncthreads_and(ok)) return fail();
  }
  // ---------------------------------------------------------------- 1. norms, gate scan
  {   // row norms: 4 threads per row, 32 channels each (word order rotated by row)
    const int r = tid >> 2, part = tid & 3, rot = 2 * (r & 7);
    const bf16 *sq_ = (const bf16 *)(smem + S::STQ), *sk_ = (const bf16 *)(smem + S::STK);
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = part * 32 + 2 * ((i + rot) & 15);
      const float2 fq = ld2(sq_ + r * D + c), fk = ld2(sk_ + r * D + c);
      sq = fmaf(fq.x, fq.x, fmaf(fq.y, fq.y, sq));
      sk = fmaf(fk.x, fk.x, fmaf(fk.y, fk.y, sk));
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
  // Channel-major pass, thread = (channels ch and 64 + ch, sub-block a): the gate scan, then (after
  // the barrier) Kh, the per-channel factor tables and the local sums cs_r = G_r - E_{a-1} (log2
  // units) in shared memory for the row-major pass. The row-major pass's raw q, k of the first
  // channel half come out of the staging here too, before the local sums overwrite it.
  const int ch = tid & 63, a = tid >> 6;
  const int q8 = tid & 7, rb = tid >> 3;     // row-major pass: channels 32 g + 4 q8 .., rows rb and rb + 32
  uint2 qraw[4][2], kraw[4][2];              // raw q, k (4 bf16) of the row-major pass per K-block g
  {
    float cs0[SUB], cs1[SUB];
    __nv_bfloat162 kk[SUB];
    const bf16 *sq_ = (const bf16 *)(smem + S::STQ), *sk_ = (const bf16 *)(smem + S::STK);
    const float *sg = (const float *)(smem + S::STG);
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int r = rb + 32 * s2;
        qraw[g][s2] = *reinterpret_cast<const uint2 *>(sq_ + r * D + 32 * g + 4 * q8);
        kraw[g][s2] = *reinterpret_cast<const uint2 *>(sk_ + r * D + 32 * g + 4 * q8);
      }
    float run0 = 0.f, run1 = 0.f;
#pragma unroll
    for (int i = 0; i < SUB; ++i) {
      const int r = a * SUB + i;
      kk[i] = __halves2bfloat162(sk_[r * D + ch], sk_[r * D + 64 + ch]);
      run0 = fmaf(sg[r * D + ch], LOG2E, run0);
      run1 = fmaf(sg[r * D + 64 + ch], LOG2E, run1);
      cs0[i] = run0;
      cs1[i] = run1;
    }
    tot[a][ch] = run0;
    tot[a][64 + ch] = run1;
    __syncthreads();   // norms and sub-block sums in place; the q, k staging is dead from here on
    float *csm = (float *)(smem + S::CS);
    float *pam = (float *)(smem + S::PA), *pfm = (float *)(smem + S::PF);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int c = 64 * hh + ch;
      float em[NSUB + 1];   // E_{b-1} of channel c (log2), b = 0..4, summed in one fixed order
      em[0] = 0.f;
#pragma unroll
      for (int b = 0; b < NSUB; ++b) em[b + 1] = em[b] + tot[b][c];
      float ema = em[0];   // em[a], picked by compile-time indices (a run-time index would put em in local memory)
#pragma unroll
      for (int b = 1; b < NSUB; ++b)
        if (b == a) ema = em[b];
      if (a == 0) *reinterpret_cast<float *>(rec + TcRec::GC + 4 * c) = ex2(em[NSUB]);   // e^{G_last}
      pam[a * 128 + c] = ex2(ema);
#pragma unroll
      for (int ap = 1; ap < NSUB; ++ap)
        if (ap > a) pfm[pair_idx(a, ap) * 128 + c] = ex2(em[ap] - ema);
      // Kh = k^ e^{G_last - G} into the record (B2 rows 0..127, transposed: row c, tokens 16a..)
      const float ftail = em[NSUB] - ema;
#pragma unroll
      for (int i8 = 0; i8 < SUB; i8 += 8) {
        float khv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int i = i8 + e, r = a * SUB + i;
          const float csr = hh ? cs1[i] : cs0[i];
          khv[e] = (hh ? __high2float(kk[i]) : __low2float(kk[i])) * rk[r] * ex2(ftail - csr);
          csm[r * D + c] = csr;
        }
        *reinterpret_cast<uint4 *>(rec + TcRec::B2 + tc::sw128_off(192, c, a * SUB + i8)) = tc::pack8(khv);
      }
    }
  }
  __syncthreads();   // local sums and factor tables in place

  // ---------------------------------------------------------------- 2. Gram products
  // Row-major pass over the four K-blocks g of 32 channels, thread = (channels 32 g + 4 q8 ..,
  // rows rb and rb + 32): each operand row segment is one 16-byte store. K-block g goes to buffer
  // g & 1 and its product is issued at once, so it runs while the next K-block is written; a
  // buffer is rewritten once the product two K-blocks back (on bar[2 + buffer]) has read it.
  {   // the raw q, k of K-blocks 2 and 3 from global memory (rows past the sequence read 0)
#pragma unroll
    for (int g = 2; g < 4; ++g)
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int r = rb + 32 * s2;
        const size_t off = ((size_t)(ref.t0 + r) * H + h) * D + 32 * g + 4 * q8;
        const bool in = r < ref.len;
        qraw[g][s2] = in ? *reinterpret_cast<const uint2 *>((const bf16 *)p.q + off) : make_uint2(0u, 0u);
        kraw[g][s2] = in ? *reinterpret_cast<const uint2 *>((const bf16 *)p.k + off) : make_uint2(0u, 0u);
      }
  }
  float bk[4][2][4];   // Diag(beta) Kt of this thread's rows and channels, for W's operand
  {
    const float *csm = (const float *)(smem + S::CS);
    const float *pam = (const float *)(smem + S::PA), *pfm = (const float *)(smem + S::PF);
    bool ok = true;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int bf = g & 1, c0 = 32 * g + 4 * q8;
      if (g >= 2) {   // the product of K-block g - 2 has read this buffer
        ok &= mbar_wait(&bar[2 + bf], 0);
        tc::fence_after();
      }
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int r = rb + 32 * s2, ar = r >> 4;
        const float4 cs4 = *reinterpret_cast<const float4 *>(csm + r * D + c0);
        const float4 pa4 = *reinterpret_cast<const float4 *>(pam + ar * 128 + c0);
        const float csv[4] = {cs4.x, cs4.y, cs4.z, cs4.w}, pav[4] = {pa4.x, pa4.y, pa4.z, pa4.w};
        const __nv_bfloat162 q01 = *reinterpret_cast<const __nv_bfloat162 *>(&qraw[g][s2].x),
                             q23 = *reinterpret_cast<const __nv_bfloat162 *>(&qraw[g][s2].y),
                             k01 = *reinterpret_cast<const __nv_bfloat162 *>(&kraw[g][s2].x),
                             k23 = *reinterpret_cast<const __nv_bfloat162 *>(&kraw[g][s2].y);
        const float qvv[4] = {__low2float(q01), __high2float(q01), __low2float(q23), __high2float(q23)};
        const float kvv[4] = {__low2float(k01), __high2float(k01), __low2float(k23), __high2float(k23)};
        const float rqr = rq[r], rkr = rk[r], br = sb[r];
        float kl[4], ql[4], rn[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float kh = kvv[e] * rkr;
          const float x = ex2(csv[e]);            // e^{G_r - E_{a-1}} <= 1
          kl[e] = kh * x;
          ql[e] = qvv[e] * rqr * x;
          rn[e] = kh * ex2(-csv[e]);              // k^_r e^{E_{a-1} - G_r}: the right factor of block a
          bk[g][s2][e] = br * kl[e] * pav[e];
        }
        const int kk = 32 * bf + 4 * q8;            // column inside the buffer's two K-blocks
        *reinterpret_cast<float4 *>(smem + S::GA + o32(128, r, kk)) =
            make_float4(rtf32(kl[0]), rtf32(kl[1]), rtf32(kl[2]), rtf32(kl[3]));
        *reinterpret_cast<float4 *>(smem + S::GA + o32(128, 64 + r, kk)) =
            make_float4(rtf32(ql[0]), rtf32(ql[1]), rtf32(ql[2]), rtf32(ql[3]));
        // stacked right factors of the row blocks a' >= ar: k^_r e^{E_{a'-1} - G_r}
#pragma unroll
        for (int ap = 0; ap < NSUB; ++ap) {
          if (ap < ar) continue;
          float4 f = make_float4(1.f, 1.f, 1.f, 1.f);
          if (ap > ar) f = *reinterpret_cast<const float4 *>(pfm + pair_idx(ar, ap) * 128 + c0);
          *reinterpret_cast<float4 *>(smem + S::GB + o32(160, stack_off(ap) + r, kk)) =
              make_float4(rtf32(rn[0] * f.x), rtf32(rn[1] * f.y), rtf32(rn[2] * f.z), rtf32(rn[3] * f.w));
        }
        // the record's Qt (B1 rows 0..63) and the backward's Kt: 4 channels, one 8-byte store each
        __nv_bfloat162 o01 = __floats2bfloat162_rn(ql[0] * pav[0], ql[1] * pav[1]),
                       o23 = __floats2bfloat162_rn(ql[2] * pav[2], ql[3] * pav[3]);
        *reinterpret_cast<uint2 *>(rec + TcRec::B1 + tc::sw128_off(128, r, c0)) =
            make_uint2(*reinterpret_cast<uint32_t *>(&o01), *reinterpret_cast<uint32_t *>(&o23));
        if (ktrec) {
          __nv_bfloat162 t01 = __floats2bfloat162_rn(kl[0] * pav[0], kl[1] * pav[1]),
                         t23 = __floats2bfloat162_rn(kl[2] * pav[2], kl[3] * pav[3]);
          *reinterpret_cast<uint2 *>(ktrec + tc::sw128_off(64, r, c0)) =
              make_uint2(*reinterpret_cast<uint32_t *>(&t01), *reinterpret_cast<uint32_t *>(&t23));
        }
      }
      fence_proxy_async();
      tc::fence_before();
      if (!__syncthreads_and(ok)) return fail();
      tc::fence_after();
      if (tid == 0) {
        const uint32_t s_ga = smem_u32(smem + S::GA) + 16384u * bf, s_gb = smem_u32(smem + S::GB) + 20480u * bf;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc::mma_tf32(tmem, tc::desc_sw128(s_ga + 32u * ks), tc::desc_sw128(s_gb + 32u * ks), tc::idesc_tf32(128, 160),
                       (g | ks) != 0);
        tc::commit(&bar[2 + bf]);
      }
    }
    // the last product (and with it every earlier one) has completed
    ok = mbar_wait(&bar[3], 1);
    tc::fence_after();
    if (!__syncthreads_and(ok)) return fail();
  }
  // (Diag(beta) Kt)^T for W, over the dead stacked factors: rows c, token columns r
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        *reinterpret_cast<float *>(smem + S::BKT + o32(128, 32 * g + 4 * q8 + e, rb + 32 * s2)) = bk[g][s2][e];

  // ---------------------------------------------------------------- 3. Gram read-out
  // TMEM lane m: row r = m of A (m < 64) or of B (m = 64 + r); warps w and w + 4 share a lane
  // quarter and take columns j in [0, 32) and [32, 64) of each row. Row r of block ar needs the
  // stacked columns stack_off(ar) + j, j < 16 (ar + 1); a warp's lanes 0..15 and 16..31 are rows
  // of two consecutive blocks, so it loads the column ranges of both and each lane keeps its own.
  {
    const int qd = warp & 3, js = warp >> 2;
    const bool bside = qd >= 2;
    const int r = 32 * (qd & 1) + lane, ar = r >> 4;
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
    if ((qd & 1) == 0) {          // rows 0..31: blocks 0 (cols 0..15) and 1 (cols 16..47)
      if (js == 0) {
        float x0[16], x1[16], x2[16];
        tc::ld16(tl + 0, x0);
        tc::ld16(tl + 16, x1);
        tc::ld16(tl + 32, x2);
        tc::wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          v[i] = ar == 0 ? x0[i] : x1[i];
          v[16 + i] = ar == 0 ? 0.f : x2[i];
        }
      }
    } else {                      // rows 32..63: blocks 2 (cols 48..95) and 3 (cols 96..159)
      float x0[16], x1[16], y0[16], y1[16];
      if (js == 0) {
        tc::ld16(tl + 48, x0);
        tc::ld16(tl + 64, x1);
        tc::ld16(tl + 96, y0);
        tc::ld16(tl + 112, y1);
      } else {
        tc::ld16(tl + 80, x0);
        tc::ld16(tl + 80, x1);    // (no columns for j >= 48 in block 2)
        tc::ld16(tl + 128, y0);
        tc::ld16(tl + 144, y1);
      }
      tc::wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        v[i] = ar == 2 ? x0[i] : y0[i];
        v[16 + i] = ar == 2 ? (js == 0 ? x1[i] : 0.f) : y1[i];
      }
    }
    const int j0 = 32 * js;
    if (!bside) {
      // A (j < r): the backward's copy, Diag(beta) A's diagonal blocks for the solves, and -N^T
      // (column r of it: the strictly block-lower part, zero elsewhere)
      float av[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) av[i] = j0 + i < r ? v[i] : 0.f;
      if (auxA)
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *reinterpret_cast<float4 *>(auxA + r * 64 + j0 + 4 * q4) =
              make_float4(av[4 * q4], av[4 * q4 + 1], av[4 * q4 + 2], av[4 * q4 + 3]);
      const float br = sb[r];
      float *ldg = (float *)(smem + S::LD) + (ar * 16 + (r & 15)) * 17;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int j = j0 + i;
        if ((j >> 4) == ar) ldg[j & 15] = br * av[i];
        *reinterpret_cast<float *>(smem + S::NT + o32(64, j, r)) = (j >> 4) < ar ? -br * av[i] : 0.f;
      }
    } else {
      // Bm (j <= r) into the record: B2 row 128 + r, columns j0 .. j0 + 31
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        float x8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x8[e] = j0 + 8 * cb + e <= r ? v[8 * cb + e] : 0.f;
        *reinterpret_cast<uint4 *>(rec + TcRec::B2 + tc::sw128_off(192, 128 + r, j0 + 8 * cb)) = tc::pack8(x8);
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  // ---------------------------------------------------------------- 4. diagonal blocks of T
  {
    const float *ldg = (const float *)(smem + S::LD);
    if (warp < NSUB) {
      const int ab = warp, j = lane & 15;
      float x[SUB];
#pragma unroll
      for (int i = 0; i < SUB; ++i) x[i] = (i == j) ? 1.f : 0.f;
#pragma unroll
      for (int i = 1; i < SUB; ++i) {
        float s_ = 0.f;
#pragma unroll
        for (int m = 0; m < i; ++m) s_ = fmaf(ldg[(ab * 16 + i) * 17 + m], x[m], s_);
        if (i > j) x[i] = -s_;
      }
      if (lane < SUB) {
#pragma unroll
        for (int i = 0; i < SUB; ++i) {
          *reinterpret_cast<float *>(smem + S::DD + o32(64, 16 * ab + i, 16 * ab + j)) = x[i];
          *reinterpret_cast<float *>(smem + S::DT + o32(64, 16 * ab + j, 16 * ab + i)) = x[i];
        }
      }
    } else {
      // the off-diagonal blocks of D and D^T are zero
      for (int idx = tid - 128; idx < 64 * 16; idx += 128) {
        const int r = idx >> 4, k = 4 * (idx & 15);
        if ((k >> 4) != (r >> 4)) {
          *reinterpret_cast<float4 *>(smem + S::DD + o32(64, r, k)) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4 *>(smem + S::DT + o32(64, r, k)) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }
  fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  // ---------------------------------------------------------------- 5. T by the product series
  // T = (I + E' + E'^2 + E'^3) D = F + E'^2 F with F = D + E' D, in three rounds of products:
  //   1: E' = D (-N)                          -> E' [r][m] and E'^T [j][m]
  //   2: (E' D)^T = D^T E'^T, E'^2 = E' E'     -> F^T = D^T + (E' D)^T [j][m], E'^2 [r][m]
  //   3: E'^2 F                                -> T = F + E'^2 F, row by row
  // read-out of an M = 64 result: warp w has rows 16 (w & 3) + lane (lanes 0..15) and columns
  // 32 (w >> 2) .. + 31
  const int orow = 16 * (warp & 3) + (lane & 15), ocol = 32 * (warp >> 2);
  const uint32_t s_dd = smem_u32(smem + S::DD), s_dt = smem_u32(smem + S::DT), s_nt = smem_u32(smem + S::NT),
                 s_ep = smem_u32(smem + S::EP);
  if (tid == 0) {   // E' [r][j] = sum_m D[r][m] (-N^T)[j][m]
    mma64(tmem, s_dd, s_nt, 64, 8192);
    tc::commit(&bar[1]);
  }
  if (!mma_done()) return fail();
  {   // E' rows into EP; E'^T over the dead D
    float v[32];
    ld32(tl + ocol, v);
    if (lane < 16) {
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        *reinterpret_cast<float4 *>(smem + S::EP + o32(64, orow, ocol + 4 * q4)) =
            make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
#pragma unroll
      for (int i = 0; i < 32; ++i) *reinterpret_cast<float *>(smem + S::DD + o32(64, ocol + i, orow)) = v[i];
    }
  }
  fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (tid == 0) {
    mma64(tmem, s_dt, s_ep, 64, 8192);        // (E' D)^T [j][r] = sum_m D^T[j][m] E'[r][m]
    mma64(tmem + 64, s_ep, s_dd, 64, 8192);   // E'^2 [r][j]    = sum_m E'[r][m] E'^T[j][m]
    tc::commit(&bar[1]);
  }
  if (!mma_done()) return fail();
  {   // F^T = D^T + (E' D)^T over the dead -N^T; E'^2 over the dead E'^T
    float v[32], w[32];
    ld32(tl + ocol, v);
    ld32(tl + 64 + ocol, w);
    if (lane < 16) {
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        const uint32_t o = o32(64, orow, ocol + 4 * q4);
        const float4 dt = *reinterpret_cast<const float4 *>(smem + S::DT + o);
        *reinterpret_cast<float4 *>(smem + S::NT + o) =
            make_float4(dt.x + v[4 * q4], dt.y + v[4 * q4 + 1], dt.z + v[4 * q4 + 2], dt.w + v[4 * q4 + 3]);
        *reinterpret_cast<float4 *>(smem + S::DD + o) = make_float4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
      }
    }
  }
  fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (tid == 0) {   // E'^2 F [r][j] = sum_m E'^2[r][m] F^T[j][m]
    mma64(tmem, s_dd, s_nt, 64, 8192);
    tc::commit(&bar[1]);
  }
  if (!mma_done()) return fail();
  {   // T row r = F[r][.] + (E'^2 F)[r][.] (F[r][j] = F^T[j][r]): the W operand T [r][j] over the dead
      // E', Tb = T Diag(beta) into the record and T for the backward, 16-byte stores
    float v[32];
    ld32(tl + ocol, v);
    if (lane < 16) {
      const int r = orow;
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] += *reinterpret_cast<const float *>(smem + S::NT + o32(64, ocol + i, r));
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4) {
        *reinterpret_cast<float4 *>(smem + S::EP + o32(64, r, ocol + 4 * q4)) =
            make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
        if (auxT)
          *reinterpret_cast<float4 *>(auxT + r * 64 + ocol + 4 * q4) =
              make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
      }
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        float x8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x8[e] = v[8 * cb + e] * sb[ocol + 8 * cb + e];
        *reinterpret_cast<uint4 *>(rec + TcRec::TB + tc::sw128_off(64, r, ocol + 8 * cb)) = tc::pack8(x8);
      }
    }
  }
  fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  // ---------------------------------------------------------------- 6. W = T (Diag(beta) Kt)
  if (tid == 0) {
    mma64(tmem + 128, s_ep, smem_u32(smem + S::BKT), 128, 16384);
    tc::commit(&bar[1]);
  }
  if (!mma_done()) return fail();
  {   // -W [r][c] into B1 rows 64 + r: warp w has rows 16 (w & 3) + lane, channels 64 (w >> 2) ..
    const int r = orow, c0 = 64 * (warp >> 2);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float v[32];
      ld32(tl + 128 + c0 + 32 * half, v);
      if (lane < 16) {
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          float x8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) x8[e] = -v[8 * cb + e];
          *reinterpret_cast<uint4 *>(rec + TcRec::B1 + tc::sw128_off(128, 64 + r, c0 + 32 * half + 8 * cb)) =
              tc::pack8(x8);
        }
      }
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, TCOLS);
}

cudaError_t launch_prep_tc(const PrepParams &p, cudaStream_t s) {
  if (p.geo.max_chunks == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kda_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, PtSmem::BYTES);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.geo.max_chunks * p.geo.heads;   // head-fastest: see the kernel
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  // prefetch distance: the CTAs resident at once (one wave)
  int dev = 0, sms = 0, per_sm = 0;
  PrepParams q = p;
  q.prefetch_dist = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_prep_tc_kernel, PT_THREADS, PtSmem::BYTES) == cudaSuccess)
    q.prefetch_dist = sms * per_sm;
  kda_prep_tc_kernel<<<(unsigned)blocks, PT_THREADS, PtSmem::BYTES, s>>>(q);
  return cudaGetLastError();
}

}  // namespace kda
