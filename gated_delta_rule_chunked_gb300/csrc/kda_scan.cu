// kda_scan.cu -- the sequential inter-chunk state passing for fp32 I/O (the
// bf16 forward and the backward dS scan run on tcgen05, kda_scan_tc.cu).
//
// Columns of the state evolve independently (the decay and the erase act on key
// rows), so the value dimension is cut into slices of DVS columns, each an
// independent chain run by one group of 4 warps (NG groups per CTA share one
// fetched record; the fp32 path launches NG = 1). The state slice stays in
// registers for the whole sequence; its copy in shared memory is the operand of
// the fp32 products. The next chunk's values are loaded one chunk ahead into
// registers. Per chunk, with the record written
// by the prep kernel (Qt = q^*exp(G), Kt = k^*exp(G), Kh = k^*exp(G_last - G),
// Tb = T Diag(beta), Bm = masked gated q.k^T, gC = exp(G_last)):
//
//   V' = V - Kt S;  U = Tb V';  O = Qt S + Bm U;  S <- gC*S + Kh^T U
//
// (V' is the value minus what the decayed state already predicts; U is the
// delta-rule update after the intra-chunk WY/UT transform.) The record of the
// next chunk is fetched with TMA bulk copies into the regions that the current
// chunk has finished with, tracked by four mbarriers.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

template <typename E, int DVS, int NG>
struct ScanSmem {
  static constexpr int T128 = 64 * 128 * (int)sizeof(E), T64 = 64 * 64 * (int)sizeof(E);
  // record regions (same byte layout as ImgLayout)
  static constexpr int QT = 0, KT = T128, TB = 2 * T128, BM = TB + T64, KH = BM + T64, GC = KH + T128;
  static constexpr int REC = GC + 512;
  static constexpr int R1 = QT, R1B = 2 * T128;     // Qt, Kt
  static constexpr int R2 = TB, R2B = T64;          // Tb
  static constexpr int R3 = BM, R3B = T64;          // Bm
  static constexpr int R4 = KH, R4B = T128 + 512;   // Kh, gC
  static constexpr int SL = DVS * (int)sizeof(E);   // bytes per slice row
  static constexpr int GRP = 128 * SL + 3 * 64 * SL;   // per-group tiles
  static constexpr int G0 = (REC + 127) / 128 * 128;
  // per group g at G0 + g*GRP: [128][DVS] state / dS operand, then three [64][DVS] tiles
  static constexpr int X0 = 0, X1 = 128 * SL, X2 = X1 + 64 * SL, X3 = X2 + 64 * SL;
  static constexpr int BAR = G0 + NG * GRP;
  static constexpr int BYTES = BAR + 64;
};

__device__ __forceinline__ void issue_region(char *smem, const char *rec, int off, int bytes, uint64_t *bar) {
  fence_proxy_async();
  mbar_expect_tx(bar, bytes);
  bulk_g2s(smem + off, rec + off, bytes, bar);
}

// Element offset of (row, col) in a swizzled 128x128 E tile (saved-state records).
template <typename E>
__device__ __forceinline__ size_t full_off(int r, int c) {
  constexpr int EPC = 16 / sizeof(E), CPR = 128 / EPC;
  return (size_t)r * 128 + swz<CPR>(r, c / EPC) * EPC + (c % EPC);
}

// ------------------------------------------------------------------ forward
template <typename E, int DVS, int NG>
__global__ void __launch_bounds__(128 * NG, 1) kda_fwd_scan_kernel(FwdScanParams p) {
  constexpr int NZ = 128 / DVS, NT = DVS / 8, NB = NZ / NG;
  using S = ScanSmem<E, DVS, NG>;
  extern __shared__ __align__(128) char smem[];
  const int H = p.geo.heads;
  const int tid = threadIdx.x, lane = tid & 31, g8 = lane >> 2, q4 = lane & 3;
  const int grp = tid >> 7, warp = (tid >> 5) & 3;   // value-slice group, warp within the group
  const int z = (blockIdx.x % NB) * NG + grp, h = (blockIdx.x / NB) % H, seq = blockIdx.x / (NB * H);
  const long long s0 = p.geo.cu[seq], s1 = p.geo.cu[seq + 1];
  const int nch = (int)((s1 - s0 + CH - 1) / CH), cbase = p.geo.chunk_off[seq];
  char *gsm = smem + S::G0 + grp * S::GRP;
  const size_t rec_bytes = (size_t)S::REC;
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::BAR);
  Tile<E, 128> Qt((E *)(smem + S::QT)), Kt((E *)(smem + S::KT)), Kh((E *)(smem + S::KH));
  Tile<E, 64> Tb((E *)(smem + S::TB)), Bm((E *)(smem + S::BM));
  const float *gC = (const float *)(smem + S::GC);
  Tile<E, DVS> sS((E *)(gsm + S::X0)), sVp((E *)(gsm + S::X1)), sU((E *)(gsm + S::X2)), sO((E *)(gsm + S::X3));
  const E *v = (const E *)p.v;
  E *o = (E *)p.o;
  // value fragment loader (rows 16*warp + g8 + 8*hh, columns z*DVS + 8*nt + 2*q4)
  auto load_v = [&](int j, float2 (&vf)[NT][2]) {
    const long long t0 = s0 + (long long)j * CH;
    const int clen = (int)(s1 - t0 < CH ? s1 - t0 : CH);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = 16 * warp + g8 + 8 * hh;
        vf[nt][hh] = make_float2(0.f, 0.f);   // v == NULL: zero values
        if (r < clen && v) vf[nt][hh] = ld2(v + ((size_t)(t0 + r) * H + h) * 128 + z * DVS + 8 * nt + 2 * q4);
      }
  };

  // state slice: rows c = 32*warp + 16*mt + g8 + 8*hh, columns z*DVS + 8*nt + 2*q4 (+1)
  float accS[2][NT][4];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int c = 32 * warp + 16 * mt + g8 + 8 * hh, vv = z * DVS + 8 * nt + 2 * q4;
        float2 x = make_float2(0.f, 0.f);
        if (p.h0_identity) x = make_float2(c == vv ? 1.f : 0.f, c == vv + 1 ? 1.f : 0.f);
        else if (p.h0) x = *reinterpret_cast<const float2 *>(p.h0 + (((size_t)seq * H + h) * 128 + c) * 128 + vv);
        accS[mt][nt][2 * hh] = x.x;
        accS[mt][nt][2 * hh + 1] = x.y;
        st2(sS.at(c, 8 * nt + 2 * q4), x.x, x.y);
      }
  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto rec_of = [&](int j) { return (const char *)p.img + ((size_t)(cbase + j) * H + h) * rec_bytes; };
  if (tid == 0 && nch > 0) {
    const char *r0 = rec_of(0);
    issue_region(smem, r0, S::R1, S::R1B, &bar[0]);
    issue_region(smem, r0, S::R2, S::R2B, &bar[1]);
    issue_region(smem, r0, S::R3, S::R3B, &bar[2]);
    issue_region(smem, r0, S::R4, S::R4B, &bar[3]);
  }
  bool ok = true;
  float2 vnext[NT][2];
  if (nch > 0) load_v(0, vnext);
  for (int j = 0; j < nch; ++j) {
    const uint32_t par = j & 1;
    const long long t0 = s0 + (long long)j * CH;
    const int clen = (int)(s1 - t0 < CH ? s1 - t0 : CH);
    float2 vf[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) { vf[nt][0] = vnext[nt][0]; vf[nt][1] = vnext[nt][1]; }
    if (j + 1 < nch) load_v(j + 1, vnext);   // one chunk ahead
    // chunk-start state for the backward
    if (p.saved) {
      E *sv = (E *)p.saved + ((size_t)(cbase + j) * H + h) * 128 * 128;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int c = 32 * warp + 16 * mt + g8 + 8 * hh, vv = z * DVS + 8 * nt + 2 * q4;
            st2(sv + full_off<E>(c, vv), accS[mt][nt][2 * hh], accS[mt][nt][2 * hh + 1]);
          }
    }
    // (a) V' = V - Kt S ;  O = Qt S
    ok &= mbar_wait(&bar[0], par);
    float accV[NT][4], accO[NT][4];
    zero(accV);
    zero(accO);
    wgemm2<NT>(accV, accO, Kt, Qt, 16 * warp, sS, 0, 0, 128);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        st2(sVp.at(16 * warp + g8 + 8 * hh, 8 * nt + 2 * q4), vf[nt][hh].x - accV[nt][2 * hh],
            vf[nt][hh].y - accV[nt][2 * hh + 1]);
    if (!__syncthreads_and(ok)) { report(p.status, ERR_TIMEOUT); return; }
    if (tid == 0 && j + 1 < nch) issue_region(smem, rec_of(j + 1), S::R1, S::R1B, &bar[0]);
    // (b) U = Tb V'   (Tb lower triangular)
    ok &= mbar_wait(&bar[1], par);
    float accU[NT][4];
    zero(accU);
    wgemm<true, false, NT>(accU, Tb, 16 * warp, sVp, 0, 0, 16 * (warp + 1));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        st2(sU.at(16 * warp + g8 + 8 * hh, 8 * nt + 2 * q4), accU[nt][2 * hh], accU[nt][2 * hh + 1]);
    if (!__syncthreads_and(ok)) { report(p.status, ERR_TIMEOUT); return; }
    if (tid == 0 && j + 1 < nch) issue_region(smem, rec_of(j + 1), S::R2, S::R2B, &bar[1]);
    // (c) O += Bm U
    ok &= mbar_wait(&bar[2], par);
    wgemm<true, false, NT>(accO, Bm, 16 * warp, sU, 0, 0, 16 * (warp + 1));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        st2(sO.at(16 * warp + g8 + 8 * hh, 8 * nt + 2 * q4), accO[nt][2 * hh], accO[nt][2 * hh + 1]);
    // (d) S <- gC * S + Kh^T U
    ok &= mbar_wait(&bar[3], par);
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const float d0 = gC[32 * warp + 16 * mt + g8], d1 = gC[32 * warp + 16 * mt + g8 + 8];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        accS[mt][nt][0] *= d0; accS[mt][nt][1] *= d0;
        accS[mt][nt][2] *= d1; accS[mt][nt][3] *= d1;
      }
      wgemm<false, false, NT>(accS[mt], Kh, 32 * warp + 16 * mt, sU, 0, 0, 64);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
          st2(sS.at(32 * warp + 16 * mt + g8 + 8 * hh, 8 * nt + 2 * q4), accS[mt][nt][2 * hh],
              accS[mt][nt][2 * hh + 1]);
    }
    if (!__syncthreads_and(ok)) { report(p.status, ERR_TIMEOUT); return; }
    // output rows, 16-byte coalesced
    {
      constexpr int EPC = 16 / sizeof(E), CPR = DVS / EPC;
      for (int idx = tid & 127; idx < 64 * CPR; idx += 128) {
        const int r = idx / CPR, ch = idx % CPR;
        if (r < clen && o)   // o == NULL: no outputs
          *reinterpret_cast<uint4 *>(o + ((size_t)(t0 + r) * H + h) * 128 + z * DVS + ch * EPC) =
              *reinterpret_cast<const uint4 *>(sO.at(r, ch * EPC));
      }
    }
    if (tid == 0 && j + 1 < nch) {
      issue_region(smem, rec_of(j + 1), S::R3, S::R3B, &bar[2]);
      issue_region(smem, rec_of(j + 1), S::R4, S::R4B, &bar[3]);
    }
  }
  if (p.hT) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int c = 32 * warp + 16 * mt + g8 + 8 * hh, vv = z * DVS + 8 * nt + 2 * q4;
          *reinterpret_cast<float2 *>(p.hT + (((size_t)seq * H + h) * 128 + c) * 128 + vv) =
              make_float2(accS[mt][nt][2 * hh], accS[mt][nt][2 * hh + 1]);
        }
  }
}

template <typename K>
static cudaError_t launch_scan_kernel(K kern, int bytes, unsigned grid, int threads, const void *params,
                                      cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  void *args[] = {const_cast<void *>(params)};
  return cudaLaunchKernel((const void *)kern, dim3(grid), dim3(threads), args, bytes, s);
}

// fp32 I/O: one 4-warp CTA per 32-column slice of each (sequence, head). The bf16
// forward runs on the tcgen05 scan (kda_scan_tc.cu).
cudaError_t launch_fwd_scan(const FwdScanParams &p, bool f32, int, cudaStream_t s) {
  const long long units = (long long)p.geo.n_seqs * p.geo.heads;
  if (units == 0) return cudaSuccess;
  if (!f32) return cudaErrorNotSupported;
  return launch_scan_kernel(kda_fwd_scan_kernel<float, 32, 1>, ScanSmem<float, 32, 1>::BYTES,
                            (unsigned)(units * 4), 128, &p, s);
}

}  // namespace kda
