// kda_bwd.cu -- chunk-parallel parts of the KDA backward.
//
// The reverse dS scan (kda_scan.cu) leaves, for every chunk, the state
// gradient dS at the chunk end and the value gradient. Two chunk-parallel
// kernels then finish the chunk-local gradients:
//
//  state kernel (per chunk, head), with the forward's chunk-start state S and the
//  chunk-end state gradient dS (both kept transposed, [v][k], as the scans produce them):
//     V' = V - Kt S,  U = Tb V',  dU = Bm^T dO + Kh dS,  dV' = Tb^T dU
//     dQt = dO S^T,   dKt = -dV' S^T,  dKh = U dS^T,
//     dBm = dO U^T (j <= r),  dTb = dU V'^T (j <= r),  dgC_c = sum_v S_cv dS_cv
//
//  intra kernel (per chunk, head): back through the intra-chunk graph
//     Tb = T Diag(beta),  T = (I + Diag(beta) A)^-1:
//        dT = dTb Diag(beta),  dL = -T^T dT T^T,  dA = Diag(beta) dL (strict lower)
//     A, Bm through the bounded gating factors (the factorisation of kda_prep.cu),
//     Qt, Kt, Kh, gC through exp(G), then dg = reverse cumulative sum of dG
//     inside the chunk, and the L2-norm backward for q and k.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

// ------------------------------------------------------------ state kernel
constexpr int STATE_THREADS = 512;   // 16 warps: 4 row blocks x 4 column quarters of every product

template <typename E>
struct StateSmem {
  static constexpr int T128 = 64 * 128 * (int)sizeof(E), T64 = 64 * 64 * (int)sizeof(E);
  // the backward record's BMT, KH (contiguous), TBT, GC (contiguous) and KT, packed
  static constexpr int BMT = 0, KH = BMT + T64, TBT = KH + T128, GC = TBT + T64, KT = GC + 1024;
  static constexpr int REC = KT + T128;
  static constexpr int SS = (REC + 127) / 128 * 128;      // S^T [128][128]
  static constexpr int SDS = SS + 2 * T128;               // dS^T [128][128]
  static constexpr int SV = SDS + 2 * T128;               // V -> V' [64][128]
  static constexpr int SDO = SV + T128;
  static constexpr int SU = SDO + T128;
  static constexpr int SDU = SU + T128;
  static constexpr int SDV = SDU + T128;                  // -dV'
  static constexpr int BAR = SDV + T128;
  static constexpr int BYTES = BAR + 16;
};

template <typename E>
__global__ void __launch_bounds__(STATE_THREADS) kda_bwd_state_kernel(BwdStateParams p) {
  using S = StateSmem<E>;
  extern __shared__ __align__(128) char smem[];
  const int chunk = blockIdx.x, h = blockIdx.y, H = p.geo.heads;
  ChunkRef ref;
  if (!chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, chunk, ref)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, q4 = lane & 3;
  const int mt = warp & 3, nq = warp >> 2;   // 16-row block, 32-column quarter
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::BAR);
  const size_t rid = (size_t)chunk * H + h;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    fence_proxy_async();
    const char *rb = (const char *)p.img + rid * TcRecB::BYTES;
    mbar_expect_tx(bar, (TcRecB::QWT - TcRecB::BMT) + (TcRecB::SCAN - TcRecB::TBT) + S::T128 + 4 * S::T128);
    bulk_g2s(smem + S::BMT, rb + TcRecB::BMT, TcRecB::QWT - TcRecB::BMT, bar);     // Bm^T, Kh
    bulk_g2s(smem + S::TBT, rb + TcRecB::TBT, TcRecB::SCAN - TcRecB::TBT, bar);    // Tb^T, e^{G_last}
    bulk_g2s(smem + S::KT, rb + TcRecB::KT, S::T128, bar);                          // Kt
    bulk_g2s(smem + S::SS, (const char *)p.saved + rid * 2 * S::T128, 2 * S::T128, bar);
    bulk_g2s(smem + S::SDS, (const char *)p.dsaved + rid * 2 * S::T128, 2 * S::T128, bar);
  }
  // operand tiles in the tcgen05 swizzled layout the prep wrote them in
  TileSW<64> Kt((bf16 *)(smem + S::KT)), Kh((bf16 *)(smem + S::KH)), TbT((bf16 *)(smem + S::TBT)),
      BmT((bf16 *)(smem + S::BMT));
  // saved S^T and dS^T [v][k] arrive in the scans' operand-tile layout
  TileSW<128> sS((bf16 *)(smem + S::SS)), sdS((bf16 *)(smem + S::SDS));
  Tile<E, 128> sV((E *)(smem + S::SV)), sdO((E *)(smem + S::SDO)), sU((E *)(smem + S::SU)), sdU((E *)(smem + S::SDU)),
      sdV((E *)(smem + S::SDV));
  {
    constexpr int EPC = 16 / sizeof(E), CPR = 128 / EPC;
    const E *v = (const E *)p.v, *dO = (const E *)p.dO;
    for (int idx = tid; idx < 64 * CPR; idx += STATE_THREADS) {
      const int r = idx / CPR, ch = idx % CPR;
      uint4 a = make_uint4(0, 0, 0, 0), b = a;
      if (r < ref.len) {
        const size_t off = ((size_t)(ref.t0 + r) * H + h) * 128 + ch * EPC;
        a = __ldg(reinterpret_cast<const uint4 *>(v + off));
        b = __ldg(reinterpret_cast<const uint4 *>(dO + off));
      }
      *reinterpret_cast<uint4 *>(sV.at(r, ch * EPC)) = a;
      *reinterpret_cast<uint4 *>(sdO.at(r, ch * EPC)) = b;
    }
  }
  const bool ok = mbar_wait(bar, 0);
  if (!__syncthreads_and(ok)) { report(p.status, ERR_TIMEOUT); return; }

  float acc[4][4];
  const int r0 = 16 * mt + g8;
  // V' = V - Kt S (in place); B(k, n) = S[k][n] = S^T[n][k]
  zero(acc);
  wgemm<true, true, 4>(acc, Kt, 16 * mt, sS, 32 * nq, 0, 128);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      E *e = sV.at(r0 + 8 * hh, 32 * nq + 8 * nt + 2 * q4);
      const float2 x = ld2(e);
      st2(e, x.x - acc[nt][2 * hh], x.y - acc[nt][2 * hh + 1]);
    }
  __syncthreads();
  // U = Tb V' ;  dU = Bm^T dO + Kh dS
  zero(acc);
  wgemm<false, false, 4>(acc, TbT, 16 * mt, sV, 32 * nq, 0, 16 * (mt + 1));   // A(r, j) = Tb[r][j] = TbT[j][r]
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      st2(sU.at(r0 + 8 * hh, 32 * nq + 8 * nt + 2 * q4), acc[nt][2 * hh], acc[nt][2 * hh + 1]);
  zero(acc);
  wgemm<true, false, 4>(acc, BmT, 16 * mt, sdO, 32 * nq, 16 * mt, 64);     // A(r, j) = Bm[j][r] = BmT[r][j]
  wgemm<true, true, 4>(acc, Kh, 16 * mt, sdS, 32 * nq, 0, 128);   // B(k=c, n=v) = dS^T[v][c]
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      st2(sdU.at(r0 + 8 * hh, 32 * nq + 8 * nt + 2 * q4), acc[nt][2 * hh], acc[nt][2 * hh + 1]);
  __syncthreads();
  float *rec = p.grad + rid * (GradLayout::bytes / 4);
  // -dV' = -Tb^T dU ;  dBm = dO U^T ;  dTb = dU V'^T
  zero(acc);
  wgemm<true, false, 4>(acc, TbT, 16 * mt, sdU, 32 * nq, 16 * mt, 64);     // A(r, j) = Tb[j][r] = TbT[r][j]
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      st2(sdV.at(r0 + 8 * hh, 32 * nq + 8 * nt + 2 * q4), -acc[nt][2 * hh], -acc[nt][2 * hh + 1]);
  {
    float a4[2][4];
    zero(a4);
    wgemm<true, true, 2>(a4, sdO, 16 * mt, sU, 16 * nq, 0, 128);
    bf16 *dbm = reinterpret_cast<bf16 *>(reinterpret_cast<char *>(rec) + GradLayout::dbm);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = r0 + 8 * hh, j = 16 * nq + 8 * nt + 2 * q4;
        st2(dbm + r * 64 + j, j <= r ? a4[nt][2 * hh] : 0.f, j + 1 <= r ? a4[nt][2 * hh + 1] : 0.f);
      }
    zero(a4);
    wgemm<true, true, 2>(a4, sdU, 16 * mt, sV, 16 * nq, 0, 128);
    float *dtb = rec + GradLayout::dtb / 4;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = r0 + 8 * hh, j = 16 * nq + 8 * nt + 2 * q4;
        *reinterpret_cast<float2 *>(dtb + r * 64 + j) =
            make_float2(j <= r ? a4[nt][2 * hh] : 0.f, j + 1 <= r ? a4[nt][2 * hh + 1] : 0.f);
      }
  }
  __syncthreads();
  // dQt = dO S^T ; dKh = U dS^T ; dKt = -dV' S^T
  auto store128 = [&](size_t off, float(&a)[4][4]) {   // bf16 [64][128] at byte offset off
    bf16 *dst = reinterpret_cast<bf16 *>(reinterpret_cast<char *>(rec) + off);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        *reinterpret_cast<__nv_bfloat162 *>(dst + (r0 + 8 * hh) * 128 + 32 * nq + 8 * nt + 2 * q4) =
            __floats2bfloat162_rn(a[nt][2 * hh], a[nt][2 * hh + 1]);
  };
  zero(acc);
  wgemm<true, false, 4>(acc, sdO, 16 * mt, sS, 32 * nq, 0, 128);   // B(k=v, n=c) = S^T[v][c]
  store128(GradLayout::dqt, acc);
  zero(acc);
  wgemm<true, false, 4>(acc, sU, 16 * mt, sdS, 32 * nq, 0, 128);  // B(k=v, n=c) = dS^T[v][c]
  store128(GradLayout::dkh, acc);
  zero(acc);
  wgemm<true, false, 4>(acc, sdV, 16 * mt, sS, 32 * nq, 0, 128);
  store128(GradLayout::dkt, acc);
  {   // dgC_c = sum_v S[c][v] dS[c][v] = sum_v S^T[v][c] dS^T[v][c]: four threads per channel,
      // four independent partial sums each, quarters combined through shared memory (the V tile is free)
    const int c = tid & 127, qv = tid >> 7;
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int vv = 32 * qv; vv < 32 * qv + 32; vv += 4)
#pragma unroll
      for (int u = 0; u < 4; ++u) s4[u] = fmaf(to_f(*sS.at(vv + u, c)), to_f(*sdS.at(vv + u, c)), s4[u]);
    float *xch = reinterpret_cast<float *>(smem + S::SV);
    xch[qv * 128 + c] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    __syncthreads();
    if (qv == 0) rec[GradLayout::dgc / 4 + c] = (xch[c] + xch[128 + c]) + (xch[256 + c] + xch[384 + c]);
  }

}

// ------------------------------------------------------------ intra kernel
// Per (chunk, head), 16 warps. Inputs: q, k, g, beta; the forward's A (strict
// lower) and T from the prep run; the state-side gradients. The gating enters
// through three factor tiles (r in sub-block a, x_r = e^{G_r-E_{a-1}},
// y_r = e^{E_a-G_r}):  QL = q^ x,  KL = k^ x,  R = k^ y, and the record tiles
// Qt = QL P_a, Kt = KL P_a, Kh = R F_a (P_a = e^{E_{a-1}}, F_a = e^{E_3-E_a}).
// Gradients w.r.t. the factor tiles are gathered first, then
//   dq^ = dQL x,  dk^ = dKL x + dR y,  dG = dQL QL + dKL KL - dR R,
// dg = reverse cumulative sum of dG inside the chunk (plus the e^{G_last} terms
// on the last row), and the L2-norm backward gives dq, dk. The products through T
// (64x64) run on TF32 tensor cores; the factor tiles, dA and dBm are bf16 operands
// of the bf16 tensor cores (fp32 accumulation).
constexpr int INTRA_THREADS = 512;
constexpr int LDI = 132;   // padded fp32 row, 128-wide tiles
constexpr int LDJ = 68;    // padded fp32 row, 64-wide tiles

struct IntraSmem {
  static constexpr int T128 = 64 * LDI * 4, T64 = 64 * LDJ * 4, B128 = 64 * 128 * 2, B64 = 64 * 64 * 2;
  static constexpr int KL = 0, QL = B128, R = 2 * B128;        // bf16 factor tiles, Tile<bf16, 128>
  static constexpr int CS = 3 * B128;                          // fp32 [64][LDI]: g, local gate sums, then dG
  static constexpr int TT = CS + T128, DT = TT + T64, X = DT + T64;   // fp32 [64][LDJ]: T, dTb -> dT, X
  static constexpr int DAB = X + T64, DBB = DAB + B64;         // bf16 Tile<bf16, 64>: dA, dBm
  static constexpr int DV = DBB + B64;                         // [10][128] pair factors
  static constexpr int TOT = DV + 10 * 512;                    // [4][128]
  static constexpr int PV = TOT + 4 * 512, FV = PV + 4 * 512;  // [4][128] each
  static constexpr int RQ = FV + 4 * 512, RQ0 = RQ + 256, RK = RQ0 + 256, BETA = RK + 256;
  static constexpr int DB1 = BETA + 256, DB2 = DB1 + 256;      // dbeta parts: [64], [4][64]
  static constexpr int ROWQ = DB2 + 1024, ROWK = ROWQ + 1024;  // [4][64]
  static constexpr int PART = ROWK + 1024;                     // [4][128]
  static constexpr int DGC = PART + 2048;                      // [128]
  static constexpr int BYTES = DGC + 512;
};

// acc[nt] (16 x 8*NT) += A * B over k in [k0, k1) (multiples of 8), TF32 tensor cores.
// A(m, k) = a_ptr[m * a_rs + k * a_cs], B(k, n) = b_ptr[k * b_rs + n * b_cs] * (bscale ? bscale[n] : 1).
template <int NT>
__device__ __forceinline__ void mma_tf32_block(float (&acc)[NT][4], const float *a_ptr, int a_rs, int a_cs,
                                               const float *b_ptr, int b_rs, int b_cs, int k0, int k1,
                                               const float *bscale = nullptr) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  for (int kk = k0; kk < k1; kk += 8) {
    uint32_t a[4];
    a[0] = tf32(a_ptr[g * a_rs + (kk + q) * a_cs]);
    a[1] = tf32(a_ptr[(g + 8) * a_rs + (kk + q) * a_cs]);
    a[2] = tf32(a_ptr[g * a_rs + (kk + q + 4) * a_cs]);
    a[3] = tf32(a_ptr[(g + 8) * a_rs + (kk + q + 4) * a_cs]);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = 8 * nt + g;
      float b0 = b_ptr[(kk + q) * b_rs + n * b_cs], b1 = b_ptr[(kk + q + 4) * b_rs + n * b_cs];
      if (bscale) { b0 *= bscale[n]; b1 *= bscale[n]; }
      mma1688(acc[nt], a, tf32(b0), tf32(b1));
    }
  }
}

__global__ void __launch_bounds__(INTRA_THREADS, 1) kda_bwd_intra_kernel(BwdIntraParams p) {
  using S = IntraSmem;
  extern __shared__ __align__(128) char smem[];
  const int chunk = blockIdx.x, h = blockIdx.y, H = p.geo.heads;
  ChunkRef ref;
  if (!chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, chunk, ref)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
  const size_t rid = (size_t)chunk * H + h;
  const float *rec = p.grad + rid * (GradLayout::bytes / 4);
  const float *auxA = p.aux + rid * (2 * 64 * 64), *auxT = auxA + 64 * 64;
  const bf16 *qg = (const bf16 *)p.q, *kg = (const bf16 *)p.k;
  const Tile<bf16, 128> KLt((bf16 *)(smem + S::KL)), QLt((bf16 *)(smem + S::QL)), Rt((bf16 *)(smem + S::R));
  const Tile<bf16, 64> DAt((bf16 *)(smem + S::DAB)), DBt((bf16 *)(smem + S::DBB));
  float *CS = (float *)(smem + S::CS);
  float *TT = (float *)(smem + S::TT), *DT = (float *)(smem + S::DT), *XX = (float *)(smem + S::X);
  float(*dv)[128] = (float(*)[128])(smem + S::DV);
  float(*tot)[128] = (float(*)[128])(smem + S::TOT);
  float(*pv)[128] = (float(*)[128])(smem + S::PV);
  float(*fv)[128] = (float(*)[128])(smem + S::FV);
  float *rq = (float *)(smem + S::RQ), *rq0 = (float *)(smem + S::RQ0), *rk = (float *)(smem + S::RK),
        *sb = (float *)(smem + S::BETA);

  // P0: stage the chunk's inputs with one batch of asynchronous copies: q (bf16) in
  //     the X tile, k in the KL tile, g (fp32, row stride LDI) in the CS tile, T and
  //     dTb in their fp32 64x64 tiles, dBm (bf16) in its tile, dgC. Rows past the
  //     sequence end read as zero.
  const bf16 *sq_ = (const bf16 *)XX, *sk_ = (const bf16 *)(smem + S::KL);
  {
    const char *grec = reinterpret_cast<const char *>(rec);
    for (int idx = tid; idx < 64 * 16; idx += INTRA_THREADS) {
      const int r = idx >> 4, ch = idx & 15;
      const bool ok = r < ref.len;
      const size_t off = ok ? ((size_t)(ref.t0 + r) * H + h) * D + 8 * ch : 0;
      cp_async16((bf16 *)XX + r * D + 8 * ch, qg + off, ok ? 16 : 0);
      cp_async16((bf16 *)(smem + S::KL) + r * D + 8 * ch, kg + off, ok ? 16 : 0);
      cp_async16(TT + r * LDJ + 4 * ch, auxT + r * 64 + 4 * ch);
      cp_async16(DT + r * LDJ + 4 * ch, rec + GradLayout::dtb / 4 + r * 64 + 4 * ch);
      if (ch < 8) cp_async16(DBt.at(r, 8 * ch), grec + GradLayout::dbm + r * 128 + 16 * ch);
    }
    for (int idx = tid; idx < 64 * 32; idx += INTRA_THREADS) {
      const int r = idx >> 5, ch = idx & 31;
      const bool ok = r < ref.len;
      const float *src = ok ? p.g + ((size_t)(ref.t0 + r) * H + h) * D + 4 * ch : p.g;
      cp_async16(CS + r * LDI + 4 * ch, src, ok ? 16 : 0);
    }
    if (tid < 32) cp_async16((float *)(smem + S::DGC) + 4 * tid, rec + GradLayout::dgc / 4 + 4 * tid);
    if (tid < 64) sb[tid] = tid < ref.len ? p.beta[(size_t)(ref.t0 + tid) * H + h] : 0.f;
    cp_async_wait_all();
  }
  __syncthreads();
  // P1: row norms (8 threads per row)
  {
    const int r = tid >> 3, part = tid & 7;
    float sq = 0.f, sk = 0.f;
#pragma unroll
    for (int c = 0; c < 16; c += 2) {
      const float2 a = ld2(sq_ + r * D + part * 16 + c), b = ld2(sk_ + r * D + part * 16 + c);
      sq = fmaf(a.x, a.x, fmaf(a.y, a.y, sq));
      sk = fmaf(b.x, b.x, fmaf(b.y, b.y, sk));
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if (part == 0) {
      const float r0 = rsqrtf(sq + 1e-6f);
      rq0[r] = r0;
      rq[r] = p.scale * r0;
      rk[r] = rsqrtf(sk + 1e-6f);
    }
  }
  // P2a: gate scan (threads 0..255: channel pair x sub-block); this thread's raw q, k pairs
  const int cp = tid & 63, a = (tid >> 6) & 3, c0 = 2 * cp;
  float2 cs[SUB];
  __nv_bfloat162 qpair[SUB], kpair[SUB];
  if (tid < 256) {
#pragma unroll
    for (int i = 0; i < SUB; ++i) {
      const int r = a * SUB + i;
      cs[i] = *reinterpret_cast<const float2 *>(CS + r * LDI + c0);
      qpair[i] = *reinterpret_cast<const __nv_bfloat162 *>(sq_ + r * D + c0);
      kpair[i] = *reinterpret_cast<const __nv_bfloat162 *>(sk_ + r * D + c0);
    }
    float2 run = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < SUB; ++i) {
      run.x = fmaf(cs[i].x, LOG2E, run.x);
      run.y = fmaf(cs[i].y, LOG2E, run.y);
      cs[i] = run;
    }
    tot[a][c0] = run.x;
    tot[a][c0 + 1] = run.y;
  }
  __syncthreads();
  if (tid < 256) {
    // P2b: factor tiles and per-channel factors
    float em[2] = {0.f, 0.f}, e3[2] = {0.f, 0.f}, eb[2] = {0.f, 0.f};
#pragma unroll
    for (int b = 0; b < NSUB; ++b) {
      const float t0 = tot[b][c0], t1 = tot[b][c0 + 1];
      if (b < a) { em[0] += t0; em[1] += t1; }
      e3[0] += t0;
      e3[1] += t1;
    }
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
    const float ta0 = tot[a][c0], ta1 = tot[a][c0 + 1];
    pv[a][c0] = exp2f(em[0]);
    pv[a][c0 + 1] = exp2f(em[1]);
    fv[a][c0] = exp2f(e3[0] - em[0] - ta0);
    fv[a][c0 + 1] = exp2f(e3[1] - em[1] - ta1);
#pragma unroll
    for (int i = 0; i < SUB; ++i) {
      const int r = a * SUB + i;
      const float2 qv = __bfloat1622float2(qpair[i]), kv = __bfloat1622float2(kpair[i]);
      const float x0 = exp2f(cs[i].x), x1 = exp2f(cs[i].y);
      const float y0 = exp2f(ta0 - cs[i].x), y1 = exp2f(ta1 - cs[i].y);
      const float kh0 = kv.x * rk[r], kh1 = kv.y * rk[r];
      st2(KLt.at(r, c0), kh0 * x0, kh1 * x1);
      st2(QLt.at(r, c0), qv.x * rq[r] * x0, qv.y * rq[r] * x1);
      st2(Rt.at(r, c0), kh0 * y0, kh1 * y1);
      *reinterpret_cast<float2 *>(CS + r * LDI + c0) = cs[i];
    }
  } else if (tid < 320) {
    // dbeta_j through Tb = T Diag(beta), and dT = dTb Diag(beta)
    const int j = tid - 256;
    float sacc = 0.f;
    for (int r = j; r < 64; ++r) {
      const float d = DT[r * LDJ + j];
      sacc = fmaf(d, TT[r * LDJ + j], sacc);
      DT[r * LDJ + j] = d * sb[j];
    }
    ((float *)(smem + S::DB1))[j] = sacc;
  }
  __syncthreads();
  // P3: X = dT T^T (dT, T lower triangular)
  {
    const int mt = warp & 3, np = warp >> 2;     // rows 16mt.., columns 16np..16np+15
    float acc[2][4];
    zero(acc);
    mma_tf32_block<2>(acc, DT + 16 * mt * LDJ, LDJ, 1, TT + 16 * np * LDJ, 1, LDJ, 0, 16 * (mt + 1));
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float *dst = XX + (16 * mt + g) * LDJ + 16 * np + 8 * nt + 2 * q;
      *reinterpret_cast<float2 *>(dst) = make_float2(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<float2 *>(dst + 8 * LDJ) = make_float2(acc[nt][2], acc[nt][3]);
    }
  }
  __syncthreads();
  // P4: dL = -T^T X (strict lower part);  dA = Diag(beta) dL;  dbeta_r += sum_j dL_rj A_rj
  {
    const int mt = warp & 3, np = warp >> 2;
    float acc[2][4];
    zero(acc);
    mma_tf32_block<2>(acc, TT + 16 * mt, 1, LDJ, XX + 16 * np, LDJ, 1, 16 * mt, 64);
    float part[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * mt + g + 8 * hh, j = 16 * np + 8 * nt + 2 * q;
        const float d0 = j < r ? -acc[nt][2 * hh] : 0.f, d1 = j + 1 < r ? -acc[nt][2 * hh + 1] : 0.f;
        const float2 av = *reinterpret_cast<const float2 *>(auxA + r * 64 + j);
        part[hh] = fmaf(d0, j < r ? av.x : 0.f, fmaf(d1, j + 1 < r ? av.y : 0.f, part[hh]));
        st2(DAt.at(r, j), sb[r] * d0, sb[r] * d1);
      }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      part[hh] += __shfl_xor_sync(0xffffffffu, part[hh], 1);
      part[hh] += __shfl_xor_sync(0xffffffffu, part[hh], 2);
      if (q == 0) ((float *)(smem + S::DB2))[np * 64 + 16 * mt + g + 8 * hh] = part[hh];
    }
  }
  __syncthreads();
  // The 64x64 tiles T and X are dead from here on: stage q and k again (for the
  // epilogue and the L2-norm backward) while the factor-tile products run.
  const bf16 *eq_ = (const bf16 *)XX, *ek_ = (const bf16 *)TT;
  for (int idx = tid; idx < 64 * 16; idx += INTRA_THREADS) {
    const int r = idx >> 4, ch = idx & 15;
    const bool ok = r < ref.len;
    const size_t off = ok ? ((size_t)(ref.t0 + r) * H + h) * D + 8 * ch : 0;
    cp_async16((bf16 *)XX + r * D + 8 * ch, qg + off, ok ? 16 : 0);
    cp_async16((bf16 *)TT + r * D + 8 * ch, kg + off, ok ? 16 : 0);
  }
  // P5: gradients w.r.t. the factor tiles; warp -> (row sub-block t, channel quarter cq)
  const int t = warp & 3, cq = warp >> 2, cbase = 32 * cq;
  // this thread's elements of the state-side gradients dQt, dKt, dKh, loaded now so the
  // loads are in flight during the products
  __nv_bfloat162 gq[4][2], gk[4][2], gh[4][2];
  {
    const bf16 *gqt = reinterpret_cast<const bf16 *>(reinterpret_cast<const char *>(rec) + GradLayout::dqt);
    const bf16 *gkt = reinterpret_cast<const bf16 *>(reinterpret_cast<const char *>(rec) + GradLayout::dkt);
    const bf16 *gkh = reinterpret_cast<const bf16 *>(reinterpret_cast<const char *>(rec) + GradLayout::dkh);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * t + g + 8 * hh, c = cbase + 8 * nt + 2 * q;
        gq[nt][hh] = *reinterpret_cast<const __nv_bfloat162 *>(gqt + r * 128 + c);
        gk[nt][hh] = *reinterpret_cast<const __nv_bfloat162 *>(gkt + r * 128 + c);
        gh[nt][hh] = *reinterpret_cast<const __nv_bfloat162 *>(gkh + r * 128 + c);
      }
  }
  float tQ[4][4], tK[4][4], tW[4][4];
  zero(tQ);
  zero(tK);
  zero(tW);
  // tQ, tK: sum over sub-blocks b <= t of (dBm | dA)[t, b] (R_b o D_tb); the per-channel pair
  // factor D_tb scales result columns, so each block product is scaled as it is added
  for (int b = 0; b <= t; ++b) {
    const float *dsc = dv[t * (t + 1) / 2 + b] + cbase;
    float pq[4][4], pk[4][4];
    zero(pq);
    zero(pk);
    wgemm<true, false, 4>(pq, DBt, 16 * t, Rt, cbase, 16 * b, 16 * b + 16);
    wgemm<true, false, 4>(pk, DAt, 16 * t, Rt, cbase, 16 * b, 16 * b + 16);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float d = dsc[8 * nt + 2 * q + (e & 1)];
        tQ[nt][e] = fmaf(pq[nt][e], d, tQ[nt][e]);
        tK[nt][e] = fmaf(pk[nt][e], d, tK[nt][e]);
      }
  }
  // tW: sum over sub-blocks aa >= t of D_{aa,t} o ((dBm^T QL + dA^T KL)[aa rows -> t])
  for (int aa = t; aa < NSUB; ++aa) {
    float tR[4][4];
    zero(tR);
    wgemm<false, false, 4>(tR, DBt, 16 * t, QLt, cbase, 16 * aa, 16 * aa + 16);
    wgemm<false, false, 4>(tR, DAt, 16 * t, KLt, cbase, 16 * aa, 16 * aa + 16);
    const float *dsc = dv[aa * (aa + 1) / 2 + t] + cbase;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) tW[nt][e] = fmaf(tR[nt][e], dsc[8 * nt + 2 * q + (e & 1)], tW[nt][e]);
  }
  cp_async_wait_all();
  __syncthreads();   // every warp is done reading the factor tiles of other rows; q, k staged
  float dqh[4][4], dkh[4][4];
  {
    float rowq[2] = {0.f, 0.f}, rowk[2] = {0.f, 0.f}, colsum[4][2];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      colsum[nt][0] = colsum[nt][1] = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * t + g + 8 * hh, c = cbase + 8 * nt + 2 * q;
        const float2 dqt = __bfloat1622float2(gq[nt][hh]), dkt = __bfloat1622float2(gk[nt][hh]),
                     dkk = __bfloat1622float2(gh[nt][hh]);
        const float2 qr = ld2(eq_ + r * D + c), kr = ld2(ek_ + r * D + c);
        const float dqtv[2] = {dqt.x, dqt.y}, dktv[2] = {dkt.x, dkt.y}, dkkv[2] = {dkk.x, dkk.y};
        const float qrv[2] = {qr.x, qr.y}, krv[2] = {kr.x, kr.y};
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int cc = c + e2, e = 2 * hh + e2;
          const float pa = pv[t][cc], fa = fv[t][cc];
          const float csv = CS[r * LDI + cc];
          const float x = exp2f(csv), y = exp2f(tot[t][cc] - csv);
          const float ql = to_f(*QLt.at(r, cc)), kl = to_f(*KLt.at(r, cc)), rr = to_f(*Rt.at(r, cc));
          const float dQL = tQ[nt][e] + dqtv[e2] * pa, dKL = tK[nt][e] + dktv[e2] * pa;
          const float dR = tW[nt][e] + dkkv[e2] * fa;
          const float dq_ = dQL * x, dk_ = dKL * x + dR * y;
          CS[r * LDI + cc] = dQL * ql + dKL * kl - dR * rr;   // dG (natural-log units)
          colsum[nt][e2] = fmaf(dkkv[e2], rr * fa, colsum[nt][e2]);
          dqh[nt][e] = dq_;
          dkh[nt][e] = dk_;
          rowq[hh] = fmaf(qrv[e2] * rq0[r], dq_, rowq[hh]);
          rowk[hh] = fmaf(krv[e2] * rk[r], dk_, rowk[hh]);
        }
      }
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      rowq[hh] += __shfl_xor_sync(0xffffffffu, rowq[hh], 1);
      rowq[hh] += __shfl_xor_sync(0xffffffffu, rowq[hh], 2);
      rowk[hh] += __shfl_xor_sync(0xffffffffu, rowk[hh], 1);
      rowk[hh] += __shfl_xor_sync(0xffffffffu, rowk[hh], 2);
      if (q == 0) {
        ((float *)(smem + S::ROWQ))[cq * 64 + 16 * t + g + 8 * hh] = rowq[hh];
        ((float *)(smem + S::ROWK))[cq * 64 + 16 * t + g + 8 * hh] = rowk[hh];
      }
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        float sum = colsum[nt][e2];
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        sum += __shfl_xor_sync(0xffffffffu, sum, 8);
        sum += __shfl_xor_sync(0xffffffffu, sum, 16);
        if (g == 0) ((float *)(smem + S::PART))[t * 128 + cbase + 8 * nt + 2 * q + e2] = sum;
      }
  }
  __syncthreads();
  // P6: L2-norm backward, dg (reverse cumulative sum), dbeta
  {
    const float *rowQ = (const float *)(smem + S::ROWQ), *rowK = (const float *)(smem + S::ROWK);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * t + g + 8 * hh, c = cbase + 8 * nt + 2 * q;
        if (r < ref.len) {
          const size_t off = ((size_t)(ref.t0 + r) * H + h) * D + c;
          const float2 qr = ld2(eq_ + r * D + c), kr = ld2(ek_ + r * D + c);
          const float dq_dot = rowQ[r] + rowQ[64 + r] + rowQ[128 + r] + rowQ[192 + r];
          const float dk_dot = rowK[r] + rowK[64 + r] + rowK[128 + r] + rowK[192 + r];
          const float sq = p.scale * rq0[r], rkr = rk[r];
          *reinterpret_cast<float2 *>(p.dq + off) =
              make_float2(sq * (dqh[nt][2 * hh] - qr.x * rq0[r] * dq_dot),
                          sq * (dqh[nt][2 * hh + 1] - qr.y * rq0[r] * dq_dot));
          *reinterpret_cast<float2 *>(p.dk + off) =
              make_float2(rkr * (dkh[nt][2 * hh] - kr.x * rkr * dk_dot),
                          rkr * (dkh[nt][2 * hh + 1] - kr.y * rkr * dk_dot));
        }
      }
    if (tid < 128) {
      const int c = tid;
      const float *part = (const float *)(smem + S::PART);
      float e3 = tot[0][c] + tot[1][c] + tot[2][c] + tot[3][c];
      float run = part[c] + part[128 + c] + part[256 + c] + part[384 + c] +
                  ((const float *)(smem + S::DGC))[c] * exp2f(e3);
      for (int r = 63; r >= 0; --r) {
        run += CS[r * LDI + c];
        if (r < ref.len) p.dg[((size_t)(ref.t0 + r) * H + h) * 128 + c] = run;
      }
    } else if (tid < 192) {
      const int r = tid - 128;
      const float *d2 = (const float *)(smem + S::DB2);
      if (r < ref.len)
        p.dbeta[(size_t)(ref.t0 + r) * H + h] =
            ((const float *)(smem + S::DB1))[r] + d2[r] + d2[64 + r] + d2[128 + r] + d2[192 + r];
    }
  }
}

template <typename K>
static cudaError_t launch_chunk_kernel(K kern, int bytes, dim3 grid, int threads, const void *params,
                                       cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  void *args[] = {const_cast<void *>(params)};
  return cudaLaunchKernel((const void *)kern, grid, dim3(threads), args, bytes, s);
}

cudaError_t launch_bwd_state(const BwdStateParams &p, bool f32, cudaStream_t s) {
  if (p.geo.max_chunks == 0) return cudaSuccess;
  if (f32) return cudaErrorNotSupported;
  return launch_chunk_kernel(kda_bwd_state_kernel<bf16>, StateSmem<bf16>::BYTES,
                             dim3(p.geo.max_chunks, p.geo.heads), STATE_THREADS, &p, s);
}

cudaError_t launch_bwd_intra(const BwdIntraParams &p, bool f32, cudaStream_t s) {
  if (p.geo.max_chunks == 0) return cudaSuccess;
  if (f32) return cudaErrorNotSupported;
  return launch_chunk_kernel(kda_bwd_intra_kernel, IntraSmem::BYTES, dim3(p.geo.max_chunks, p.geo.heads),
                             INTRA_THREADS, &p, s);
}

}  // namespace kda
