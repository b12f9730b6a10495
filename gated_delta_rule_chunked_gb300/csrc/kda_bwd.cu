// kda_bwd.cu -- chunk-parallel parts of the KDA backward.
//
// The reverse dS scan (kda_scan.cu) leaves, for every chunk, the state
// gradient dS at the chunk end and the value gradient. Two chunk-parallel
// kernels then finish the chunk-local gradients:
//
//  state kernel (per chunk, head), with the forward's chunk-start state S:
//     V' = V - Kt S,  U = Tb V',  dU = Bm^T dO + Kh dS,  dV' = Tb^T dU
//     dQt = dO S^T,   dKt = -dV' S^T,  dKh = U dS^T,
//     dBm = dO U^T (j <= r),  dTb = dU V'^T (j <= r),  dgC_c = sum_v S_cv dS_cv
//
//  intra kernel (per chunk, head): back through the intra-chunk graph
//     Tb = T Diag(beta),  T = (I + Diag(beta) A)^-1:
//        dT = dTb Diag(beta),  dL = -T^T dT T^T,  dA = Diag(beta) dL (strict lower)
//     A, Bm through the bounded gating factors (see kda_intra.cuh),
//     Qt, Kt, Kh, gC through exp(G), then dg = reverse cumulative sum of dG
//     inside the chunk, and the L2-norm backward for q and k.
#include "kda_common.cuh"
#include "kda_intra.cuh"
#include "kda_internal.h"

namespace kda {

// ------------------------------------------------------------ state kernel
template <typename E>
struct StateSmem {
  static constexpr int T128 = 64 * 128 * (int)sizeof(E), T64 = 64 * 64 * (int)sizeof(E);
  static constexpr int QT = 0, KT = T128, TB = 2 * T128, BM = TB + T64, KH = BM + T64, GC = KH + T128;
  static constexpr int REC = GC + 512;
  static constexpr int SS = (REC + 127) / 128 * 128;      // S  [128][128]
  static constexpr int SDS = SS + 2 * T128;               // dS [128][128]
  static constexpr int SV = SDS + 2 * T128;               // V -> V' [64][128]
  static constexpr int SDO = SV + T128;
  static constexpr int SU = SDO + T128;
  static constexpr int SDU = SU + T128;
  static constexpr int SDV = SDU + T128;                  // -dV'
  static constexpr int BAR = SDV + T128;
  static constexpr int BYTES = BAR + 16;
};

template <typename E>
__global__ void __launch_bounds__(256) kda_bwd_state_kernel(BwdStateParams p) {
  using S = StateSmem<E>;
  extern __shared__ __align__(128) char smem[];
  const int chunk = blockIdx.x, h = blockIdx.y, H = p.geo.heads;
  ChunkRef ref;
  if (!chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, chunk, ref)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, q4 = lane & 3;
  const int mt = warp & 3, nh = warp >> 2;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::BAR);
  const size_t rid = (size_t)chunk * H + h;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    fence_proxy_async();
    mbar_expect_tx(bar, S::REC + 4 * S::T128);
    bulk_g2s(smem, (const char *)p.img + rid * S::REC, S::REC, bar);
    bulk_g2s(smem + S::SS, (const char *)p.saved + rid * 2 * S::T128, 2 * S::T128, bar);
    bulk_g2s(smem + S::SDS, (const char *)p.dsaved + rid * 2 * S::T128, 2 * S::T128, bar);
  }
  Tile<E, 128> Kt((E *)(smem + S::KT)), Kh((E *)(smem + S::KH));
  Tile<E, 64> Tb((E *)(smem + S::TB)), Bm((E *)(smem + S::BM));
  Tile<E, 128> sS((E *)(smem + S::SS)), sdS((E *)(smem + S::SDS)), sV((E *)(smem + S::SV)),
      sdO((E *)(smem + S::SDO)), sU((E *)(smem + S::SU)), sdU((E *)(smem + S::SDU)), sdV((E *)(smem + S::SDV));
  {
    constexpr int EPC = 16 / sizeof(E), CPR = 128 / EPC;
    const E *v = (const E *)p.v, *dO = (const E *)p.dO;
    for (int idx = tid; idx < 64 * CPR; idx += 256) {
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

  float acc[8][4];
  const int r0 = 16 * mt + g8;
  // V' = V - Kt S (in place)
  zero(acc);
  wgemm<true, false, 8>(acc, Kt, 16 * mt, sS, 64 * nh, 0, 128);
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      E *e = sV.at(r0 + 8 * hh, 64 * nh + 8 * nt + 2 * q4);
      const float2 x = ld2(e);
      st2(e, x.x - acc[nt][2 * hh], x.y - acc[nt][2 * hh + 1]);
    }
  __syncthreads();
  // U = Tb V' ;  dU = Bm^T dO + Kh dS
  zero(acc);
  wgemm<true, false, 8>(acc, Tb, 16 * mt, sV, 64 * nh, 0, 16 * (mt + 1));
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      st2(sU.at(r0 + 8 * hh, 64 * nh + 8 * nt + 2 * q4), acc[nt][2 * hh], acc[nt][2 * hh + 1]);
  zero(acc);
  wgemm<false, false, 8>(acc, Bm, 16 * mt, sdO, 64 * nh, 16 * mt, 64);
  wgemm<true, false, 8>(acc, Kh, 16 * mt, sdS, 64 * nh, 0, 128);
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      st2(sdU.at(r0 + 8 * hh, 64 * nh + 8 * nt + 2 * q4), acc[nt][2 * hh], acc[nt][2 * hh + 1]);
  __syncthreads();
  float *rec = p.grad + rid * (GradLayout::bytes / 4);
  // -dV' = -Tb^T dU ;  dBm = dO U^T ;  dTb = dU V'^T
  zero(acc);
  wgemm<false, false, 8>(acc, Tb, 16 * mt, sdU, 64 * nh, 16 * mt, 64);
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      st2(sdV.at(r0 + 8 * hh, 64 * nh + 8 * nt + 2 * q4), -acc[nt][2 * hh], -acc[nt][2 * hh + 1]);
  {
    float a4[4][4];
    zero(a4);
    wgemm<true, true, 4>(a4, sdO, 16 * mt, sU, 32 * nh, 0, 128);
    float *dbm = rec + GradLayout::dbm / 4;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = r0 + 8 * hh, j = 32 * nh + 8 * nt + 2 * q4;
        *reinterpret_cast<float2 *>(dbm + r * 64 + j) =
            make_float2(j <= r ? a4[nt][2 * hh] : 0.f, j + 1 <= r ? a4[nt][2 * hh + 1] : 0.f);
      }
    zero(a4);
    wgemm<true, true, 4>(a4, sdU, 16 * mt, sV, 32 * nh, 0, 128);
    float *dtb = rec + GradLayout::dtb / 4;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = r0 + 8 * hh, j = 32 * nh + 8 * nt + 2 * q4;
        *reinterpret_cast<float2 *>(dtb + r * 64 + j) =
            make_float2(j <= r ? a4[nt][2 * hh] : 0.f, j + 1 <= r ? a4[nt][2 * hh + 1] : 0.f);
      }
  }
  __syncthreads();
  // dQt = dO S^T ; dKh = U dS^T ; dKt = -dV' S^T
  auto store128 = [&](float *dst, float(&a)[8][4]) {
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        *reinterpret_cast<float2 *>(dst + (r0 + 8 * hh) * 128 + 64 * nh + 8 * nt + 2 * q4) =
            make_float2(a[nt][2 * hh], a[nt][2 * hh + 1]);
  };
  zero(acc);
  wgemm<true, true, 8>(acc, sdO, 16 * mt, sS, 64 * nh, 0, 128);
  store128(rec + GradLayout::dqt / 4, acc);
  zero(acc);
  wgemm<true, true, 8>(acc, sU, 16 * mt, sdS, 64 * nh, 0, 128);
  store128(rec + GradLayout::dkh / 4, acc);
  zero(acc);
  wgemm<true, true, 8>(acc, sdV, 16 * mt, sS, 64 * nh, 0, 128);
  store128(rec + GradLayout::dkt / 4, acc);
  if (tid < 128) {
    float s = 0.f;
    for (int vv = 0; vv < 128; vv += 2) {
      const float2 a = ld2(sS.at(tid, vv)), b = ld2(sdS.at(tid, vv));
      s = fmaf(a.x, b.x, fmaf(a.y, b.y, s));
    }
    rec[GradLayout::dgc / 4 + tid] = s;
  }
}

// ------------------------------------------------------------ intra kernel
template <typename E>
struct IntraSmem {
  using P = PrepSmem<E>;
  static constexpr int W0 = (P::BYTES + 127) / 128 * 128;   // A (fp32 64x64) ; later dG (with W1)
  static constexpr int W1 = W0 + 16384;                     // Lm -> X
  static constexpr int W2 = W1 + 16384;                     // T
  static constexpr int W3 = W2 + 16384;                     // dTb -> dT
  static constexpr int DA = W3 + 16384;                     // dA (E 64x64)
  static constexpr int DB = DA + 64 * 64 * (int)sizeof(E);  // dBm (E 64x64)
  static constexpr int SCR = DB + 64 * 64 * (int)sizeof(E); // 4 KB
  static constexpr int DB1 = SCR + 4096, DB2 = DB1 + 256;   // dbeta parts [64]
  static constexpr int ROWQ = DB2 + 256, ROWK = ROWQ + 512; // [2][64]
  static constexpr int PART = ROWK + 512;                   // [4][128]
  static constexpr int DGC = PART + 2048;                   // [128]
  static constexpr int BYTES = DGC + 512;
};

template <typename E>
__global__ void __launch_bounds__(256) kda_bwd_intra_kernel(BwdIntraParams p) {
  using P = PrepSmem<E>;
  using S = IntraSmem<E>;
  extern __shared__ __align__(128) char smem[];
  const int chunk = blockIdx.x, h = blockIdx.y, H = p.geo.heads;
  ChunkRef ref;
  if (!chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, chunk, ref)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, q4 = lane & 3;
  const size_t rid = (size_t)chunk * H + h;
  const float *rec = p.grad + rid * (GradLayout::bytes / 4);
  Tile<float, 64> tA((float *)(smem + S::W0)), tLm((float *)(smem + S::W1)), tT((float *)(smem + S::W2)),
      tdT((float *)(smem + S::W3)), tX((float *)(smem + S::W1));
  Tile<E, 64> tdA((E *)(smem + S::DA)), tdB((E *)(smem + S::DB));
  const float *sb = (const float *)(smem + P::BETA);

  load_chunk_qkg<E>(smem, (const E *)p.q, (const E *)p.k, p.g, p.beta, ref.t0, ref.len, h, H, 256);
  for (int idx = tid; idx < 64 * 32; idx += 256) {
    const int r = idx / 32, j = (idx % 32) * 2;
    const float2 a = *reinterpret_cast<const float2 *>(rec + GradLayout::dtb / 4 + r * 64 + j);
    const float2 b = *reinterpret_cast<const float2 *>(rec + GradLayout::dbm / 4 + r * 64 + j);
    st2(tdT.at(r, j), a.x, a.y);
    st2(tdB.at(r, j), b.x, b.y);
  }
  if (tid < 128) ((float *)(smem + S::DGC))[tid] = rec[GradLayout::dgc / 4 + tid];
  __syncthreads();
  row_norms<E>(smem, p.scale);
  gate_scan<E>(smem);
  __syncthreads();
  factor_pass<E>(smem);
  __syncthreads();
  // A (strict lower): warps 0..3 own row sub-block a' = warp
  if (warp < NSUB) {
    const int ap = warp;
    Tile<E, 128> tk((E *)(smem + P::K));
#pragma unroll
    for (int b = 0; b < NSUB; ++b) {
      float accA[2][4];
      zero(accA);
      if (b <= ap) {
        Tile<E, 128> rd((E *)(smem + P::RD) + pair_idx(ap, b) * SUB * 128);
        wgemm<true, true, 2>(accA, tk, ap * SUB, rd, 0, 0, 128);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = ap * SUB + g8 + 8 * hh, j = b * SUB + nt * 8 + 2 * q4;
          const float a0 = (j < r) ? accA[nt][2 * hh] : 0.f, a1 = (j + 1 < r) ? accA[nt][2 * hh + 1] : 0.f;
          st2(tA.at(r, j), a0, a1);
          st2(tLm.at(r, j), sb[r] * a0, sb[r] * a1);
        }
    }
  }
  __syncthreads();
  ut_solve((float *)(smem + S::W1), (float *)(smem + S::W2), (float *)(smem + S::SCR));
  // dbeta_j (through Tb = T Diag(beta)) and dT = dTb Diag(beta)
  if (tid < 64) {
    const int j = tid;
    float s = 0.f;
    for (int r = j; r < 64; ++r) {
      const float d = *tdT.at(r, j);
      s = fmaf(d, *tT.at(r, j), s);
      *tdT.at(r, j) = d * sb[j];
    }
    ((float *)(smem + S::DB1))[j] = s;
  }
  __syncthreads();
  // X = dT T^T
  {
    const int r = tid >> 2, m0 = (tid & 3) * 16;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = 0.f;
    for (int j = 0; j <= r; ++j) {
      const float d = *tdT.at(r, j);
#pragma unroll
      for (int i = 0; i < 16; ++i) x[i] = fmaf(d, *tT.at(m0 + i, j), x[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; i += 2) st2(tX.at(r, m0 + i), x[i], x[i + 1]);
  }
  __syncthreads();
  // dL = -T^T X (strict lower);  dA = Diag(beta) dL ;  dbeta_r += sum_j dL_rj A_rj
  {
    const int r = tid >> 2, j0 = (tid & 3) * 16;
    float dl[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) dl[i] = 0.f;
    for (int m = r; m < 64; ++m) {
      const float t = *tT.at(m, r);
#pragma unroll
      for (int i = 0; i < 16; ++i) dl[i] = fmaf(t, *tX.at(m, j0 + i), dl[i]);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
      const int j = j0 + i;
      const float d0 = (j < r) ? -dl[i] : 0.f, d1 = (j + 1 < r) ? -dl[i + 1] : 0.f;
      s = fmaf(d0, *tA.at(r, j), fmaf(d1, *tA.at(r, j + 1), s));
      st2(tdA.at(r, j), sb[r] * d0, sb[r] * d1);
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    if ((tid & 3) == 0) ((float *)(smem + S::DB2))[r] = s;
  }
  __syncthreads();

  // Gram backward and gate combine: warp -> row sub-block t, channel half hf
  const int t = warp & 3, hf = warp >> 2;
  Tile<E, 128> QL((E *)(smem + P::Q)), KL((E *)(smem + P::K));
  Tile<float, 128> tG((float *)(smem + P::G)), tdG((float *)(smem + S::W0));
  const float(*ev)[128] = (const float(*)[128])(smem + P::EV);
  const float(*pv)[128] = (const float(*)[128])(smem + P::PV);
  const float *fv = (const float *)(smem + P::FV);
  float dqh[8][4], dkh[8][4];
  float colsum[8][2];
  float rowq[2] = {0.f, 0.f}, rowk[2] = {0.f, 0.f};
  {
    float tQ[8][4], tK[8][4], tW[8][4], dG[8][4];
    zero(tQ);
    zero(tK);
    zero(tW);
    zero(dG);
    for (int b = 0; b <= t; ++b) {
      Tile<E, 128> rdb((E *)(smem + P::RD) + (pair_idx(t, b) - b) * SUB * 128);
      wgemm<true, false, 8>(tQ, tdB, 16 * t, rdb, 64 * hf, 16 * b, 16 * b + 16);
      wgemm<true, false, 8>(tK, tdA, 16 * t, rdb, 64 * hf, 16 * b, 16 * b + 16);
    }
    for (int a = t; a < NSUB; ++a) {
      float tR[8][4];
      zero(tR);
      wgemm<false, false, 8>(tR, tdB, 16 * t, QL, 64 * hf, 16 * a, 16 * a + 16);
      wgemm<false, false, 8>(tR, tdA, 16 * t, KL, 64 * hf, 16 * a, 16 * a + 16);
      Tile<E, 128> rdat((E *)(smem + P::RD) + pair_idx(a, t) * SUB * 128);
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int jl = g8 + 8 * (e >> 1), c = 64 * hf + 8 * nt + 2 * q4 + (e & 1);
          const float dat = exp2f(ev[a][c] - ev[t + 1][c]);
          tW[nt][e] = fmaf(tR[nt][e], dat, tW[nt][e]);
          dG[nt][e] = fmaf(-tR[nt][e], to_f(*rdat.at(jl, c)), dG[nt][e]);
        }
    }
    Tile<E, 128> rd3((E *)(smem + P::RD) + pair_idx(3, 0) * SUB * 128);
    const E *qg = (const E *)p.q, *kg = (const E *)p.k;
    const float *rq0 = (const float *)(smem + P::RQ0), *rk = (const float *)(smem + P::RK);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      colsum[nt][0] = colsum[nt][1] = 0.f;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * t + g8 + 8 * hh, c = 64 * hf + 8 * nt + 2 * q4;
        const float2 dqt = *reinterpret_cast<const float2 *>(rec + GradLayout::dqt / 4 + r * 128 + c);
        const float2 dkt = *reinterpret_cast<const float2 *>(rec + GradLayout::dkt / 4 + r * 128 + c);
        const float2 dkhs = *reinterpret_cast<const float2 *>(rec + GradLayout::dkh / 4 + r * 128 + c);
        float2 qr = make_float2(0.f, 0.f), kr = qr;
        if (r < ref.len) {
          const size_t off = ((size_t)(ref.t0 + r) * H + h) * 128 + c;
          qr = ld2(qg + off);
          kr = ld2(kg + off);
        }
        const float dqv[2] = {dqt.x, dqt.y}, dktv[2] = {dkt.x, dkt.y}, dkhv[2] = {dkhs.x, dkhs.y};
        const float qrv[2] = {qr.x, qr.y}, krv[2] = {kr.x, kr.y};
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int cc = c + e2, e = 2 * hh + e2;
          const float Gr = *tG.at(r, cc);
          const float x = exp2f(Gr - ev[t][cc]), y = exp2f(ev[t + 1][cc] - Gr);
          const float px = pv[t][cc], ft = exp2f(ev[4][cc] - ev[t + 1][cc]);
          const float ql = to_f(*QL.at(r, cc)), kl = to_f(*KL.at(r, cc));
          const float khv = to_f(*rd3.at(r, cc)) * fv[cc];
          const float xq = x * px;
          const float dq_ = tQ[nt][e] * x + dqv[e2] * xq;
          const float dk_ = tK[nt][e] * x + tW[nt][e] * y + dktv[e2] * xq + dkhv[e2] * (y * ft);
          const float dg_ = dG[nt][e] + tQ[nt][e] * ql + tK[nt][e] * kl + (dqv[e2] * ql + dktv[e2] * kl) * px -
                            dkhv[e2] * khv;
          colsum[nt][e2] = fmaf(dkhv[e2], khv, colsum[nt][e2]);
          dqh[nt][e] = dq_;
          dkh[nt][e] = dk_;
          *tdG.at(r, cc) = dg_;
          rowq[hh] = fmaf(qrv[e2] * rq0[r], dq_, rowq[hh]);
          rowk[hh] = fmaf(krv[e2] * rk[r], dk_, rowk[hh]);
        }
      }
    }
  }
  // row dot products for the norm backward; column sums of dKh*Kh for dG_last
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    rowq[hh] += __shfl_xor_sync(0xffffffffu, rowq[hh], 1);
    rowq[hh] += __shfl_xor_sync(0xffffffffu, rowq[hh], 2);
    rowk[hh] += __shfl_xor_sync(0xffffffffu, rowk[hh], 1);
    rowk[hh] += __shfl_xor_sync(0xffffffffu, rowk[hh], 2);
    if (q4 == 0) {
      ((float *)(smem + S::ROWQ))[hf * 64 + 16 * t + g8 + 8 * hh] = rowq[hh];
      ((float *)(smem + S::ROWK))[hf * 64 + 16 * t + g8 + 8 * hh] = rowk[hh];
    }
  }
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int e2 = 0; e2 < 2; ++e2) {
      float s = colsum[nt][e2];
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      s += __shfl_xor_sync(0xffffffffu, s, 8);
      s += __shfl_xor_sync(0xffffffffu, s, 16);
      if (g8 == 0) ((float *)(smem + S::PART))[t * 128 + 64 * hf + 8 * nt + 2 * q4 + e2] = s;
    }
  __syncthreads();
  // dq, dk: L2-norm backward
  {
    const float *rowQ = (const float *)(smem + S::ROWQ), *rowK = (const float *)(smem + S::ROWK);
    const float *rq0 = (const float *)(smem + P::RQ0), *rk = (const float *)(smem + P::RK);
    const E *qg = (const E *)p.q, *kg = (const E *)p.k;
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * t + g8 + 8 * hh, c = 64 * hf + 8 * nt + 2 * q4;
        if (r < ref.len) {
          const size_t off = ((size_t)(ref.t0 + r) * H + h) * 128 + c;
          const float2 qr = ld2(qg + off), kr = ld2(kg + off);
          const float dq_dot = rowQ[r] + rowQ[64 + r], dk_dot = rowK[r] + rowK[64 + r];
          const float sq = p.scale * rq0[r], rkr = rk[r];
          *reinterpret_cast<float2 *>(p.dq + off) =
              make_float2(sq * (dqh[nt][2 * hh] - qr.x * rq0[r] * dq_dot),
                          sq * (dqh[nt][2 * hh + 1] - qr.y * rq0[r] * dq_dot));
          *reinterpret_cast<float2 *>(p.dk + off) =
              make_float2(rkr * (dkh[nt][2 * hh] - kr.x * rkr * dk_dot),
                          rkr * (dkh[nt][2 * hh + 1] - kr.y * rkr * dk_dot));
        }
      }
  }
  // dg = reverse cumulative sum of dG inside the chunk; dbeta
  if (tid < 128) {
    const int c = tid;
    const float *part = (const float *)(smem + S::PART);
    const float gcv = ((const float *)(smem + P::GC))[c];
    float run = part[c] + part[128 + c] + part[256 + c] + part[384 + c] + ((const float *)(smem + S::DGC))[c] * gcv;
    for (int r = 63; r >= 0; --r) {
      run += *tdG.at(r, c);
      if (r < ref.len) p.dg[((size_t)(ref.t0 + r) * H + h) * 128 + c] = run;
    }
  } else if (tid < 192) {
    const int r = tid - 128;
    if (r < ref.len)
      p.dbeta[(size_t)(ref.t0 + r) * H + h] = ((const float *)(smem + S::DB1))[r] + ((const float *)(smem + S::DB2))[r];
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
                             dim3(p.geo.max_chunks, p.geo.heads), 256, &p, s);
}

cudaError_t launch_bwd_intra(const BwdIntraParams &p, bool f32, cudaStream_t s) {
  if (p.geo.max_chunks == 0) return cudaSuccess;
  if (f32) return cudaErrorNotSupported;
  return launch_chunk_kernel(kda_bwd_intra_kernel<bf16>, IntraSmem<bf16>::BYTES,
                             dim3(p.geo.max_chunks, p.geo.heads), 256, &p, s);
}

}  // namespace kda
