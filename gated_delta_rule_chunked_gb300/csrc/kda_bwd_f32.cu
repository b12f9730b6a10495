// kda_bwd_f32.cu -- the KDA backward for fp32 I/O, in plain fp32 arithmetic on the CUDA cores.
//
// The bf16 backward runs on tcgen05 (kda_scan_tc.cu, kda_bwd_tc.cu). fp32 I/O asks for
// gradients within 1e-4 of the exact ones, which bf16 or TF32 operands do not give, so this
// path forms every product with fp32 FMAs. After a prep run (kda_prep.cu, which leaves the fp32
// chunk records and A, T in the backward's workspace) three kernels follow.
//
// 1. The reverse dS scan: one 4-warp CTA per 32-column value slice of a (sequence, head); the
//    columns of dS evolve independently, as the state's do in the forward. Per chunk, from the
//    last one back, with dS the gradient at the chunk's end:
//      dU = Bm^T dO + Kh dS,   dV' = Tb^T dU (this is dv),   dS <- Diag(gC) dS + Qt^T dO - Kt^T dV'
//    and dS is saved at every chunk end for the chunk kernels.
// 2. The state side of each (chunk, head), with S its start state (saved by the forward):
//      V' = V - Kt S,  U = Tb V',  dU and dV' as above,
//      dQt = dO S^T,  dKt = -dV' S^T,  dKh = U dS^T,  dBm = dO U^T (j <= r),  dTb = dU V'^T (j <= r),
//      dgC_c = sum_v S_cv dS_cv,
//    then through Tb = T Diag(beta) and T = (I + Diag(beta) A)^-1:
//      dT = dTb Diag(beta),  dL = -(T^T dT T^T) (strict lower),  dA = Diag(beta) dL,
//      dbeta_j = sum_r dTb_rj T_rj + sum_i dL_ji A_ji   (beta enters only through Tb and T).
//    dQt, dKt and dKh go to the dq, dk and dg arrays (the rows of this chunk), dBm, dA and
//    dgC e^{G_last} to a per-chunk scratch record.
// 3. The intra-chunk side. With E_rjc = exp(G_rc - G_jc), which is at most 1 for j <= r whatever
//    the gates,
//      Bm_rj = sum_c q^_rc k^_jc E_rjc (j <= r),   A_rj = sum_c k^_rc k^_jc E_rjc (j < r),
//      Qt = q^ e^G,  Kt = k^ e^G,  Kh = k^ e^{G_last - G},  gC = e^{G_last},
//    so each gradient of q^, k^ and G is a sum over token pairs whose factor E is formed directly
//    (no factorisation, hence no range condition on the gates). dg is the reverse cumulative sum
//    of dG within the chunk plus the terms through G_last, and the L2-norm backward
//    dx = r (dx^ - x^ (x^ . dx^)) (with the scale on q) gives dq and dk.
// The diagonal of Bm, Bm_rr = q^_r . k^_r, does not depend on the gates: its two contributions
// to dG_r cancel, so it is left out of dG and enters dq^ and dk^ directly.
//
// Waits are bounded; on a timeout the CTA reports KDA_ERR_TIMEOUT and returns.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

namespace {

// ------------------------------------------------------------------ 1. reverse dS scan
constexpr int BS_DVS = 32;   // value columns per CTA
constexpr int BS_NT = BS_DVS / 8;

struct BsSmem {
  static constexpr int T128 = 64 * 128 * 4, T64 = 64 * 64 * 4;
  // record regions, in the byte layout of the fp32 record (ImgLayout)
  static constexpr int QT = 0, KT = T128, TB = 2 * T128, BM = TB + T64, KH = BM + T64, GC = KH + T128;
  static constexpr int REC = GC + 512;
  static constexpr int R1 = QT, R1B = 2 * T128;     // Qt, Kt
  static constexpr int R2 = TB, R2B = T64;          // Tb
  static constexpr int R3 = BM, R3B = T64;          // Bm
  static constexpr int R4 = KH, R4B = T128 + 512;   // Kh, gC
  static constexpr int SL = BS_DVS * 4;             // bytes of one slice row
  // slice tiles: dS [128][DVS] (operand copy of the registers), dO, dU, dV' [64][DVS]
  static constexpr int DS = REC, DO = DS + 128 * SL, DU = DO + 64 * SL, DV = DU + 64 * SL;
  static constexpr int BAR = DV + 64 * SL;
  static constexpr int BYTES = BAR + 64;
};

__device__ __forceinline__ void bs_issue(char *smem, const char *rec, int off, int bytes, uint64_t *bar) {
  fence_proxy_async();
  mbar_expect_tx(bar, bytes);
  bulk_g2s(smem + off, rec + off, bytes, bar);
}

__global__ void __launch_bounds__(128, 1) kda_bwd_scan_f32_kernel(const __grid_constant__ BwdScanParams p) {
  using S = BsSmem;
  constexpr int NZ = 128 / BS_DVS, NT = BS_NT;
  extern __shared__ __align__(128) char smem[];
  const int H = p.geo.heads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g8 = lane >> 2, q4 = lane & 3;
  const int z = blockIdx.x % NZ, h = (blockIdx.x / NZ) % H, seq = blockIdx.x / (NZ * H);
  const long long s0 = p.geo.cu[seq], s1 = p.geo.cu[seq + 1];
  const int nch = (int)((s1 - s0 + CH - 1) / CH), cbase = p.geo.chunk_off[seq];
  const int col0 = z * BS_DVS;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::BAR);
  Tile<float, 128> Qt((float *)(smem + S::QT)), Kt((float *)(smem + S::KT)), Kh((float *)(smem + S::KH));
  Tile<float, 64> Tb((float *)(smem + S::TB)), Bm((float *)(smem + S::BM));
  const float *gC = (const float *)(smem + S::GC);
  Tile<float, BS_DVS> sDS((float *)(smem + S::DS)), sDO((float *)(smem + S::DO)), sDU((float *)(smem + S::DU)),
      sDV((float *)(smem + S::DV));
  const float *dO = (const float *)p.dO;
  // dO fragment loader: rows 16 warp + g8 + 8 hh, columns col0 + 8 nt + 2 q4 (+1); zero past the sequence
  auto load_do = [&](int j, float2 (&f)[NT][2]) {
    const long long t0 = s0 + (long long)j * CH;
    const int clen = (int)(s1 - t0 < CH ? s1 - t0 : CH);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * warp + g8 + 8 * hh;
        f[nt][hh] = make_float2(0.f, 0.f);
        if (r < clen) f[nt][hh] = ld2(dO + ((size_t)(t0 + r) * H + h) * 128 + col0 + 8 * nt + 2 * q4);
      }
  };

  // dS slice in registers: rows c = 32 warp + 16 mt + g8 + 8 hh, columns col0 + 8 nt + 2 q4 (+1)
  float accS[2][NT][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int c = 32 * warp + 16 * mt + g8 + 8 * hh, vv = col0 + 8 * nt + 2 * q4;
        float2 x = make_float2(0.f, 0.f);
        if (p.dhT) x = *reinterpret_cast<const float2 *>(p.dhT + (((size_t)seq * H + h) * 128 + c) * 128 + vv);
        accS[mt][nt][2 * hh] = x.x;
        accS[mt][nt][2 * hh + 1] = x.y;
        st2(sDS.at(c, 8 * nt + 2 * q4), x.x, x.y);
      }
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto rec_of = [&](int j) { return (const char *)p.img + ((size_t)(cbase + j) * H + h) * (size_t)S::REC; };
  if (tid == 0 && nch > 0) {
    const char *r0 = rec_of(nch - 1);
    bs_issue(smem, r0, S::R1, S::R1B, &bar[0]);
    bs_issue(smem, r0, S::R2, S::R2B, &bar[1]);
    bs_issue(smem, r0, S::R3, S::R3B, &bar[2]);
    bs_issue(smem, r0, S::R4, S::R4B, &bar[3]);
  }
  float2 dnext[NT][2];
  if (nch > 0) load_do(nch - 1, dnext);
  bool ok = true;
  int it = 0;
  for (int j = nch - 1; j >= 0; --j, ++it) {
    const uint32_t par = (uint32_t)(it & 1);
    const long long t0 = s0 + (long long)j * CH;
    const int clen = (int)(s1 - t0 < CH ? s1 - t0 : CH);
    // this chunk's dO into shared memory, the previous chunk's rows one step ahead
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) st2(sDO.at(16 * warp + g8 + 8 * hh, 8 * nt + 2 * q4), dnext[nt][hh].x, dnext[nt][hh].y);
    if (j > 0) load_do(j - 1, dnext);
    // dS at this chunk's end, for the chunk kernels
    if (p.dsaved) {
      Tile<float, 128> ds((float *)p.dsaved + ((size_t)(cbase + j) * H + h) * 128 * 128);
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            st2(ds.at(32 * warp + 16 * mt + g8 + 8 * hh, col0 + 8 * nt + 2 * q4), accS[mt][nt][2 * hh],
                accS[mt][nt][2 * hh + 1]);
    }
    __syncthreads();   // the dO tile is complete
    // (a) dU = Bm^T dO + Kh dS (rows 16 warp..; Bm_jr is zero for j < r)
    ok &= mbar_wait(&bar[2], par);
    ok &= mbar_wait(&bar[3], par);
    float accU[NT][4];
    zero(accU);
    if (ok) {
      wgemm<false, false, NT>(accU, Bm, 16 * warp, sDO, 0, 16 * warp, 64);
      wgemm<true, false, NT>(accU, Kh, 16 * warp, sDS, 0, 0, 128);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        st2(sDU.at(16 * warp + g8 + 8 * hh, 8 * nt + 2 * q4), accU[nt][2 * hh], accU[nt][2 * hh + 1]);
    if (!__syncthreads_and(ok)) {
      report(p.status, ERR_TIMEOUT);
      return;
    }
    if (tid == 0 && j > 0) bs_issue(smem, rec_of(j - 1), S::R3, S::R3B, &bar[2]);
    // (b) dV' = Tb^T dU (Tb_rj is zero for r < j); dv = dV'
    ok &= mbar_wait(&bar[1], par);
    float accV[NT][4];
    zero(accV);
    if (ok) wgemm<false, false, NT>(accV, Tb, 16 * warp, sDU, 0, 16 * warp, 64);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * warp + g8 + 8 * hh;
        st2(sDV.at(r, 8 * nt + 2 * q4), accV[nt][2 * hh], accV[nt][2 * hh + 1]);
        if (r < clen)
          *reinterpret_cast<float2 *>(p.dv + ((size_t)(t0 + r) * H + h) * 128 + col0 + 8 * nt + 2 * q4) =
              make_float2(accV[nt][2 * hh], accV[nt][2 * hh + 1]);
      }
    if (!__syncthreads_and(ok)) {
      report(p.status, ERR_TIMEOUT);
      return;
    }
    if (tid == 0 && j > 0) bs_issue(smem, rec_of(j - 1), S::R2, S::R2B, &bar[1]);
    // (c) dS <- Diag(gC) dS + Qt^T dO - Kt^T dV' (every warp finished reading the dS tile in (a))
    ok &= mbar_wait(&bar[0], par);
    if (ok) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const float d0 = gC[32 * warp + 16 * mt + g8], d1 = gC[32 * warp + 16 * mt + g8 + 8];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          accS[mt][nt][0] *= d0;
          accS[mt][nt][1] *= d0;
          accS[mt][nt][2] *= d1;
          accS[mt][nt][3] *= d1;
        }
        wgemm<false, false, NT>(accS[mt], Qt, 32 * warp + 16 * mt, sDO, 0, 0, 64);
        float accT[NT][4];
        zero(accT);
        wgemm<false, false, NT>(accT, Kt, 32 * warp + 16 * mt, sDV, 0, 0, 64);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) accS[mt][nt][e] -= accT[nt][e];
      }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          st2(sDS.at(32 * warp + 16 * mt + g8 + 8 * hh, 8 * nt + 2 * q4), accS[mt][nt][2 * hh],
              accS[mt][nt][2 * hh + 1]);
    if (!__syncthreads_and(ok)) {
      report(p.status, ERR_TIMEOUT);
      return;
    }
    if (tid == 0 && j > 0) {
      bs_issue(smem, rec_of(j - 1), S::R1, S::R1B, &bar[0]);
      bs_issue(smem, rec_of(j - 1), S::R4, S::R4B, &bar[3]);
    }
  }
  if (p.dh0) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int c = 32 * warp + 16 * mt + g8 + 8 * hh, vv = col0 + 8 * nt + 2 * q4;
          *reinterpret_cast<float2 *>(p.dh0 + (((size_t)seq * H + h) * 128 + c) * 128 + vv) =
              make_float2(accS[mt][nt][2 * hh], accS[mt][nt][2 * hh + 1]);
        }
  }
}

// ------------------------------------------------------------------ 2. state side
constexpr int BC_T = 256;   // threads of the chunk kernels
constexpr int CTA_KB = 32;   // k-block of the staged block products (K is a multiple of it)
constexpr int LDP = 129;    // padded fp32 row of the [64][128] tiles: row and column reads hit distinct banks

// acc[i][j] += sum_k A(4 tr + i, k) B(k, tc + 16 j) over k < K (a multiple of CTA_KB), for the
// 64 x 16 NJ product of the CTA (tr = tid / 16, tc = tid % 16). The operands are read through
// fa(r, k) and fb(k, n) (shared or global memory) into a staging area, CTA_KB values of k at a time.
template <int NJ, class FA, class FB>
__device__ __forceinline__ void cta_mm(float (&acc)[4][NJ], FA fa, FB fb, int K, float *st) {
  constexpr int N = 16 * NJ;
  float *sa = st, *sbm = st + 64 * (CTA_KB + 1);
  const int tid = threadIdx.x, tr = tid >> 4, tc = tid & 15;
  for (int k0 = 0; k0 < K; k0 += CTA_KB) {
    __syncthreads();   // the staging area is free (and earlier shared-memory results are visible)
    for (int idx = tid; idx < 64 * CTA_KB; idx += BC_T) {
      const int r = idx / CTA_KB, kk = idx % CTA_KB;
      sa[r * (CTA_KB + 1) + kk] = fa(r, k0 + kk);
    }
    for (int idx = tid; idx < CTA_KB * N; idx += BC_T) {
      const int kk = idx / N, n = idx % N;
      sbm[kk * N + n] = fb(k0 + kk, n);
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < CTA_KB; ++kk) {
      float av[4], bv[NJ];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = sa[(4 * tr + i) * (CTA_KB + 1) + kk];
#pragma unroll
      for (int j = 0; j < NJ; ++j) bv[j] = sbm[kk * N + tc + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < NJ; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
  }
  __syncthreads();   // every thread is done with the staging area and the operands
}

template <int NJ>
__device__ __forceinline__ void zero_acc(float (&acc)[4][NJ]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < NJ; ++j) acc[i][j] = 0.f;
}

struct BxSmem {
  static constexpr int TILE = 64 * LDP * 4;
  static constexpr int VP = 0, U = TILE, DU = 2 * TILE, DV = 3 * TILE;   // V', U, dU, dV' [64][LDP]
  static constexpr int ST = 4 * TILE;                                    // staging: A [64][KB + 1], B [KB][128]
  static constexpr int SB = ST + (64 * (CTA_KB + 1) + CTA_KB * 128) * 4; // beta [64]
  static constexpr int PART = SB + 256;                                  // dbeta partials [2][16][64]
  static constexpr int BYTES = PART + 2 * 16 * 64 * 4;
  // regions reused once their products are done
  static constexpr int DT = VP;   // dT [64][65]
  static constexpr int X = DU;    // X = dT T^T [64][65]
};

__global__ void __launch_bounds__(BC_T, 1) kda_bwd_state_f32_kernel(const __grid_constant__ BwdF32Params p) {
  using S = BxSmem;
  extern __shared__ __align__(128) char smem[];
  const int H = p.geo.heads, h = (int)(blockIdx.x % (unsigned)H), chunk = (int)(blockIdx.x / (unsigned)H);
  ChunkRef ref;
  if (!chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, chunk, ref)) return;
  const int tid = threadIdx.x, tr = tid >> 4, tc = tid & 15, len = ref.len;
  const long long t0 = ref.t0;
  const size_t rid = (size_t)chunk * H + h;
  const ImgLayout L(4);
  char *rec = (char *)p.img + rid * L.bytes;
  const Tile<float, 128> Kt((float *)(rec + L.kt)), Kh((float *)(rec + L.kh));
  const Tile<float, 64> Tb((float *)(rec + L.tb)), Bm((float *)(rec + L.bm));
  const float *gC = (const float *)(rec + L.gc);
  const Tile<float, 128> Sg(const_cast<float *>(p.saved) + rid * 128 * 128),
      dSg(const_cast<float *>(p.dsaved) + rid * 128 * 128);
  const float *Ag = p.aux + rid * 2 * 64 * 64, *Tg = Ag + 64 * 64;
  float *sc = p.scratch + rid * BWD_F32_SCRATCH;
  float *VP = (float *)(smem + S::VP), *U = (float *)(smem + S::U), *DU = (float *)(smem + S::DU),
        *DV = (float *)(smem + S::DV), *st = (float *)(smem + S::ST), *sb = (float *)(smem + S::SB),
        *part = (float *)(smem + S::PART);
  if (tid < 64) sb[tid] = tid < len ? p.beta[(size_t)(t0 + tid) * H + h] : 0.f;
  // token-major [T][H][128] inputs: the rows of this chunk, zero past them
  auto tok = [&](const float *base, int r, int c) -> float {
    return r < len ? __ldg(base + ((size_t)(t0 + r) * H + h) * 128 + c) : 0.f;
  };
  auto out_rows = [&](float *dst, const float (&acc)[4][8], float sign) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 4 * tr + i;
      if (r < len)
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[((size_t)(t0 + r) * H + h) * 128 + tc + 16 * j] = sign * acc[i][j];
    }
  };
  auto to_tile = [&](float *dst, const float (&acc)[4][8]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[(4 * tr + i) * LDP + tc + 16 * j] = acc[i][j];
  };
  float acc[4][8];
  // V' = V - Kt S
  zero_acc(acc);
  cta_mm<8>(acc, [&](int r, int k) { return *Kt.at(r, k); }, [&](int k, int n) { return *Sg.at(k, n); }, 128, st);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = tok(p.v, 4 * tr + i, tc + 16 * j) - acc[i][j];
  to_tile(VP, acc);
  // U = Tb V'
  zero_acc(acc);
  cta_mm<8>(acc, [&](int r, int k) { return *Tb.at(r, k); }, [&](int k, int n) { return VP[k * LDP + n]; }, 64, st);
  to_tile(U, acc);
  // dU = Bm^T dO + Kh dS
  zero_acc(acc);
  cta_mm<8>(acc, [&](int r, int k) { return *Bm.at(k, r); }, [&](int k, int n) { return tok(p.dO, k, n); }, 64, st);
  cta_mm<8>(acc, [&](int r, int k) { return *Kh.at(r, k); }, [&](int k, int n) { return *dSg.at(k, n); }, 128, st);
  to_tile(DU, acc);
  // dV' = Tb^T dU
  zero_acc(acc);
  cta_mm<8>(acc, [&](int r, int k) { return *Tb.at(k, r); }, [&](int k, int n) { return DU[k * LDP + n]; }, 64, st);
  to_tile(DV, acc);
  // dQt = dO S^T, dKt = -dV' S^T, dKh = U dS^T into the dq, dk, dg rows of this chunk
  zero_acc(acc);
  cta_mm<8>(acc, [&](int r, int k) { return tok(p.dO, r, k); }, [&](int k, int n) { return *Sg.at(n, k); }, 128, st);
  out_rows(p.dq, acc, 1.f);
  zero_acc(acc);
  cta_mm<8>(acc, [&](int r, int k) { return DV[r * LDP + k]; }, [&](int k, int n) { return *Sg.at(n, k); }, 128, st);
  out_rows(p.dk, acc, -1.f);
  zero_acc(acc);
  cta_mm<8>(acc, [&](int r, int k) { return U[r * LDP + k]; }, [&](int k, int n) { return *dSg.at(n, k); }, 128, st);
  out_rows(p.dg, acc, 1.f);
  // dBm = dO U^T (j <= r) into the scratch record
  float a4[4][4];
  zero_acc(a4);
  cta_mm<4>(a4, [&](int r, int k) { return tok(p.dO, r, k); }, [&](int k, int n) { return U[n * LDP + k]; }, 128, st);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = 4 * tr + i, jj = tc + 16 * j;
      sc[r * 64 + jj] = jj <= r ? a4[i][j] : 0.f;
    }
  // dTb = dU V'^T (j <= r); after it V' and dU are dead
  zero_acc(a4);
  cta_mm<4>(a4, [&](int r, int k) { return DU[r * LDP + k]; }, [&](int k, int n) { return VP[n * LDP + k]; }, 128, st);
  // dT = dTb Diag(beta) -> shared memory; dbeta through Tb: column sums of dTb o T
  float *DT = (float *)(smem + S::DT), *X = (float *)(smem + S::X);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int jj = tc + 16 * j;
    float cs = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = 4 * tr + i;
      const float d = jj <= r ? a4[i][j] : 0.f;
      DT[r * 65 + jj] = d * sb[jj];
      cs = fmaf(d, Tg[r * 64 + jj], cs);
    }
    part[tr * 64 + jj] = cs;
  }
  // X = dT T^T
  zero_acc(a4);
  cta_mm<4>(a4, [&](int r, int k) { return DT[r * 65 + k]; }, [&](int k, int n) { return Tg[n * 64 + k]; }, 64, st);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) X[(4 * tr + i) * 65 + tc + 16 * j] = a4[i][j];
  // dL = -(T^T X) (strict lower); dA = Diag(beta) dL into the scratch record; dbeta through A
  zero_acc(a4);
  cta_mm<4>(a4, [&](int r, int k) { return Tg[k * 64 + r]; }, [&](int k, int n) { return X[k * 65 + n]; }, 64, st);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 4 * tr + i;
    float rs = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int jj = tc + 16 * j;
      const float dl = jj < r ? -a4[i][j] : 0.f;
      sc[64 * 64 + r * 64 + jj] = sb[r] * dl;
      rs = fmaf(dl, Ag[r * 64 + jj], rs);
    }
    part[16 * 64 + tc * 64 + r] = rs;
  }
  // dgC_c e^{G_last}, dgC_c = sum_v S_cv dS_cv (two threads per channel)
  {
    const int c = tid >> 1, half = tid & 1;
    float s = 0.f;
    for (int v = 64 * half; v < 64 * half + 64; ++v) s = fmaf(*Sg.at(c, v), *dSg.at(c, v), s);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    if (!half) sc[2 * 64 * 64 + c] = s * gC[c];
  }
  __syncthreads();
  if (tid < len) {
    float db = 0.f;
    for (int i = 0; i < 16; ++i) db += part[i * 64 + tid];
    for (int i = 0; i < 16; ++i) db += part[16 * 64 + i * 64 + tid];
    p.dbeta[(size_t)(t0 + tid) * H + h] = db;
  }
}

// ------------------------------------------------------------------ 3. intra-chunk side
struct BySmem {
  static constexpr int T128 = 64 * 128 * 4, T64 = 64 * 64 * 4;
  // u_q = q r_q, k^ = k r_k, G (log2 units), dKh o Kh (then its exclusive prefix sums over rows)
  static constexpr int UQ = 0, KH = T128, G = 2 * T128, KHT = 3 * T128;
  static constexpr int DBM = 4 * T128, DA = DBM + T64;   // dBm, dA [64][64]
  static constexpr int RQ = DA + T64, RK = RQ + 256;    // r_q, r_k [64]
  static constexpr int DGC = RK + 256;                  // dgC e^{G_last} [128]
  static constexpr int RD = DGC + 512;                  // row dots [64][2][4]
  static constexpr int BYTES = RD + 64 * 8 * 4;
};

__global__ void __launch_bounds__(BC_T, 1) kda_bwd_intra_f32_kernel(const __grid_constant__ BwdF32Params p) {
  using S = BySmem;
  extern __shared__ __align__(128) char smem[];
  const int H = p.geo.heads, h = (int)(blockIdx.x % (unsigned)H), chunk = (int)(blockIdx.x / (unsigned)H);
  ChunkRef ref;
  if (!chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, chunk, ref)) return;
  const int tid = threadIdx.x, lane = tid & 31, len = ref.len;
  const long long t0 = ref.t0;
  const size_t rid = (size_t)chunk * H + h;
  float *uq = (float *)(smem + S::UQ), *kh = (float *)(smem + S::KH), *G = (float *)(smem + S::G),
        *kht = (float *)(smem + S::KHT), *dbm = (float *)(smem + S::DBM), *da = (float *)(smem + S::DA),
        *rq = (float *)(smem + S::RQ), *rk = (float *)(smem + S::RK), *dgc = (float *)(smem + S::DGC),
        *rd = (float *)(smem + S::RD);
  const float *sc = p.scratch + rid * BWD_F32_SCRATCH;
  const float s = p.scale;
  // stage q, k, g (zero past the chunk's rows) and the scratch record
  for (int idx = tid; idx < 64 * 32; idx += BC_T) {
    const int r = idx >> 5, c4 = (idx & 31) * 4;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a, c = a;
    if (r < len) {
      const size_t off = ((size_t)(t0 + r) * H + h) * 128 + c4;
      a = *reinterpret_cast<const float4 *>(p.q + off);
      b = *reinterpret_cast<const float4 *>(p.k + off);
      c = *reinterpret_cast<const float4 *>(p.g + off);
    }
    *reinterpret_cast<float4 *>(uq + r * 128 + c4) = a;
    *reinterpret_cast<float4 *>(kh + r * 128 + c4) = b;
    *reinterpret_cast<float4 *>(G + r * 128 + c4) = c;
  }
  for (int idx = tid; idx < 64 * 64 / 4; idx += BC_T) {
    *reinterpret_cast<float4 *>(dbm + 4 * idx) = *reinterpret_cast<const float4 *>(sc + 4 * idx);
    *reinterpret_cast<float4 *>(da + 4 * idx) = *reinterpret_cast<const float4 *>(sc + 64 * 64 + 4 * idx);
  }
  if (tid < 128) dgc[tid] = sc[2 * 64 * 64 + tid];
  __syncthreads();
  {   // row norms: 4 threads per row, 32 channels each
    const int r = tid >> 2, part = tid & 3;
    float sq = 0.f, sk = 0.f;
    for (int c = 32 * part; c < 32 * part + 32; ++c) {
      sq = fmaf(uq[r * 128 + c], uq[r * 128 + c], sq);
      sk = fmaf(kh[r * 128 + c], kh[r * 128 + c], sk);
    }
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 2);
    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
    sk += __shfl_xor_sync(0xffffffffu, sk, 2);
    if (part == 0) {
      rq[r] = rsqrtf(sq + 1e-6f);
      rk[r] = rsqrtf(sk + 1e-6f);
    }
  }
  __syncthreads();
  for (int idx = tid; idx < 64 * 128; idx += BC_T) {
    uq[idx] *= rq[idx >> 7];
    kh[idx] *= rk[idx >> 7];
  }
  if (tid < 128) {   // gate scan per channel, log2 units
    float run = 0.f;
    for (int r = 0; r < 64; ++r) {
      run = fmaf(G[r * 128 + tid], LOG2E, run);
      G[r * 128 + tid] = run;
    }
  }
  __syncthreads();
  // token pairs: thread = channel c, rows r = tid / 128 + 2 i (a warp shares its row)
  const int c = tid & 127, w4 = c >> 5;
  const float GL = G[63 * 128 + c];
  for (int i = 0; i < 32; ++i) {
    const int r = (tid >> 7) + 2 * i;
    if (r >= len) break;
    const float Gr = G[r * 128 + c], qr = s * uq[r * 128 + c], kr = kh[r * 128 + c];
    float p1 = 0.f, p2 = 0.f, p3 = 0.f;
    for (int j = 0; j < r; ++j) {   // r as the row of Bm and A
      const float e = exp2f(Gr - G[j * 128 + c]), kj = kh[j * 128 + c];
      p1 = fmaf(dbm[r * 64 + j] * e, kj, p1);
      p2 = fmaf(da[r * 64 + j] * e, kj, p2);
    }
    for (int i2 = r + 1; i2 < len; ++i2) {   // r as the column
      const float e = exp2f(G[i2 * 128 + c] - Gr);
      p3 = fmaf(e, fmaf(dbm[i2 * 64 + r], s * uq[i2 * 128 + c], da[i2 * 64 + r] * kh[i2 * 128 + c]), p3);
    }
    const size_t off = ((size_t)(t0 + r) * H + h) * 128 + c;
    const float dQt = p.dq[off], dKt = p.dk[off], dKh = p.dg[off];
    const float eG = exp2f(Gr), eL = exp2f(GL - Gr), bd = dbm[r * 64 + r];
    const float dqh = p1 + fmaf(bd, kr, dQt * eG);
    const float dkh = (p2 + p3) + fmaf(bd, qr, fmaf(dKt, eG, dKh * eL));
    // dG without the Kh term, which dg takes as sum over earlier rows of dKh o Kh (via G_last)
    const float dGp = fmaf(qr, p1, kr * (p2 - p3)) + fmaf(dQt, qr * eG, dKt * (kr * eG));
    kht[r * 128 + c] = dKh * (kr * eL);
    p.dq[off] = dqh;
    p.dk[off] = dkh;
    p.dg[off] = dGp;
    float a = uq[r * 128 + c] * dqh, b = kr * dkh;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      b += __shfl_xor_sync(0xffffffffu, b, o);
    }
    if (lane == 0) {
      rd[r * 8 + w4] = a;
      rd[r * 8 + 4 + w4] = b;
    }
  }
  __syncthreads();
  // L2-norm backward: dq = s r_q (dq^ - u_q (u_q . dq^)), dk = r_k (dk^ - k^ (k^ . dk^))
  for (int i = 0; i < 32; ++i) {
    const int r = (tid >> 7) + 2 * i;
    if (r >= len) break;
    const size_t off = ((size_t)(t0 + r) * H + h) * 128 + c;
    const float dotq = (rd[r * 8] + rd[r * 8 + 1]) + (rd[r * 8 + 2] + rd[r * 8 + 3]);
    const float dotk = (rd[r * 8 + 4] + rd[r * 8 + 5]) + (rd[r * 8 + 6] + rd[r * 8 + 7]);
    p.dq[off] = s * rq[r] * (p.dq[off] - uq[r * 128 + c] * dotq);
    p.dk[off] = rk[r] * (p.dk[off] - kh[r * 128 + c] * dotk);
  }
  // dg_r = sum_{r' >= r} dG'_r' + sum_{r' < r} dKh_r' Kh_r' + dgC e^{G_last}
  if (tid < 128) {
    float pre = 0.f;
    for (int r = 0; r < len; ++r) {
      const float x = kht[r * 128 + tid];
      kht[r * 128 + tid] = pre;
      pre += x;
    }
    float suf = 0.f;
    for (int r = len - 1; r >= 0; --r) {
      const size_t off = ((size_t)(t0 + r) * H + h) * 128 + tid;
      suf += p.dg[off];
      p.dg[off] = suf + kht[r * 128 + tid] + dgc[tid];
    }
  }
}

}  // namespace

cudaError_t launch_bwd_scan_f32(const BwdScanParams &p, cudaStream_t s) {
  const long long units = (long long)p.geo.n_seqs * p.geo.heads;
  if (units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_scan_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BsSmem::BYTES);
  if (e != cudaSuccess) return e;
  kda_bwd_scan_f32_kernel<<<(unsigned)(units * (128 / BS_DVS)), 128, BsSmem::BYTES, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_chunk_f32(const BwdF32Params &p, cudaStream_t s) {
  if (p.geo.max_chunks == 0) return cudaSuccess;
  const long long blocks = (long long)p.geo.max_chunks * p.geo.heads;   // head-fastest
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_state_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BxSmem::BYTES);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kda_bwd_intra_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, BySmem::BYTES);
  if (e != cudaSuccess) return e;
  kda_bwd_state_f32_kernel<<<(unsigned)blocks, BC_T, BxSmem::BYTES, s>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  kda_bwd_intra_f32_kernel<<<(unsigned)blocks, BC_T, BySmem::BYTES, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
