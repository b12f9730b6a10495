// kda_state_tc.cu -- state-side gradients of the backward on 5th-generation tensor cores.
//
// One CTA (8 warps) per (chunk, head). With S the chunk-start state (forward) and dS
// the chunk-end state gradient (reverse scan), both kept as S^T [v][k] tiles:
//   V' = V - Kt S,   U = Tb V',   dU = Bm^T dO + Kh dS,   dV' = Tb^T dU
//   dQt = dO S^T,   dKt = -dV' S^T,   dKh = U dS^T,
//   dBm = dO U^T (j <= r),   dTb = dU V'^T (j <= r),   dgC_c = sum_v S_cv dS_cv
// Every product runs as a tcgen05 MMA whose operands are tiles already in shared
// memory, read K-major or MN-major as each product needs (a tile of rows x 128 bytes
// in the 128-byte swizzle is K-major for one orientation and MN-major for the other),
// so nothing is transposed on the way in. Results with 128 rows (value or key
// channels) accumulate in TMEM with lane = channel; the 64 x 64 ones use M = 64.
// V' is formed on the tensor core too: -V'^T = V^T (-I) + S^T Kt^T.
//
// Three MMA groups, each followed by its epilogue (TMEM -> bf16 operand tiles or the
// gradient record):
//   A: -V'^T, dU^T, dQt^T          B: U^T, dV'^T, dTb          C: dBm, dKh^T, dKt^T
// Waits are bounded; on a timeout the CTA reports KDA_ERR_TIMEOUT, frees its tensor
// memory and returns.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc05.cuh"

namespace kda {

constexpr int ST5_THREADS = 256;

struct St5Smem {
  static constexpr int SS = 0, SDS = 32768;         // S^T, dS^T [v][k]: K-major over k, 2 blocks of 16 KB
  static constexpr int KT = 65536;                  // Kt [tok][k], 2 blocks of 8 KB
  static constexpr int BMT = 81920, KH = BMT + 8192;   // Bm^T [r][j] and Kh [tok][k]: one copy
  static constexpr int TBT = 106496;                // Tb^T [r][j] (+ e^{G_last}, unused here)
  static constexpr int V = 115712, DO = 132096;     // [tok][v] rows, K-major over v, 2 blocks of 8 KB
  static constexpr int ID = 148480;                 // -I [64][64]
  static constexpr int VPT = KT, UT = KT;           // V'^T, then U^T [v][tok] (after groups A, B)
  static constexpr int DUT = V, DVT = V;            // dU^T, then dV'^T [v][tok]
  static constexpr int STG = BMT;                   // output staging [64 r][128 c] bf16, per-warp blocks
  static constexpr int BAR = 156672, TSLOT = BAR + 64, XCH = TSLOT + 64;   // XCH: [128] fp32
  static constexpr int BYTES = XCH + 512 + 1024;    // + alignment slack
};

namespace {
// TMEM columns (512 allocated)
constexpr uint32_t T_VP = 0, T_DU = 64, T_DQ = 128, T_U = 192, T_DV = 256, T_DTB = 320, T_DBM = 384,
                   T_DKH = 448, T_DKT = 0;

__device__ __forceinline__ void ld32(uint32_t taddr, float (&v)[32]) {
  float a[16], b[16];
  tc::ld16(taddr, a);
  tc::ld16(taddr + 16, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = a[i];
    v[16 + i] = b[i];
  }
}
}  // namespace

__global__ void __launch_bounds__(ST5_THREADS, 1) kda_bwd_state_tc_kernel(BwdStateParams p) {
  using S = St5Smem;
  extern __shared__ __align__(1024) char smem_raw[];
  char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int chunk = blockIdx.x, h = blockIdx.y, H = p.geo.heads;
  ChunkRef ref;
  if (!chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, chunk, ref)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qw = warp & 3, hf = warp >> 2;          // lane quarter, column half
  const int row = 32 * qw + lane;                   // TMEM lane of this thread
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::BAR);   // [0] loads, [1..3] MMA groups
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + S::TSLOT);
  const size_t rid = (size_t)chunk * H + h;
  char *rec = reinterpret_cast<char *>(p.grad + rid * (GradLayout::bytes / 4));

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tl = tmem + ((uint32_t)(32 * qw) << 16);

  // ---------------------------------------------------------------- loads
  if (tid == 0) {
    const char *rb = (const char *)p.img + rid * TcRecB::BYTES;
    fence_proxy_async();
    mbar_expect_tx(&bar[0], 2 * 32768 + (TcRecB::QWT - TcRecB::BMT) + (TcRecB::SCAN - TcRecB::TBT) + 16384);
    bulk_g2s(smem + S::SS, (const char *)p.saved + rid * 32768, 32768, &bar[0]);
    bulk_g2s(smem + S::SDS, (const char *)p.dsaved + rid * 32768, 32768, &bar[0]);
    bulk_g2s(smem + S::BMT, rb + TcRecB::BMT, TcRecB::QWT - TcRecB::BMT, &bar[0]);   // Bm^T, Kh
    bulk_g2s(smem + S::TBT, rb + TcRecB::TBT, TcRecB::SCAN - TcRecB::TBT, &bar[0]);  // Tb^T, e^{G_last}
    bulk_g2s(smem + S::KT, rb + TcRecB::KT, 16384, &bar[0]);                          // Kt
  }
  {
    // V, dO rows into [tok][v] tiles (K-major over v, 128-byte swizzle); rows past the end are zero
    const bf16 *vg = (const bf16 *)p.v, *dog = (const bf16 *)p.dO;
    for (int idx = tid; idx < 64 * 16; idx += ST5_THREADS) {
      const int r = idx >> 4, ch = idx & 15;
      const bool ok = r < ref.len;
      const size_t off = ok ? ((size_t)(ref.t0 + r) * H + h) * 128 + 8 * ch : 0;
      const uint32_t dst = tc::sw128_off(64, r, 8 * ch);
      cp_async16(smem + S::V + dst, vg + off, ok ? 16 : 0);
      cp_async16(smem + S::DO + dst, dog + off, ok ? 16 : 0);
    }
    // -I [64][64] (rows n, K-major over k)
    for (int idx = tid; idx < 64 * 8; idx += ST5_THREADS) {
      const int r = idx >> 3, cc = idx & 7;
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      if ((r >> 3) == cc) {
        const int e = r & 7;   // element e of this chunk is the diagonal
        w[e >> 1] = (e & 1) ? 0xBF800000u : 0x0000BF80u;   // bf16 -1.0 in the high or low half
      }
      *reinterpret_cast<uint4 *>(smem + S::ID + tc::sw128_off(64, r, 8 * cc)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    cp_async_wait_all();
  }
  fence_proxy_async();
  bool ok = mbar_wait(&bar[0], 0);
  tc::fence_before();
  if (!__syncthreads_and(ok)) {
    report(p.status, ERR_TIMEOUT);
    if (warp == 0) tc::dealloc(tmem, 512);
    return;
  }
  tc::fence_after();

  const uint32_t s_ss = smem_u32(smem + S::SS), s_sds = smem_u32(smem + S::SDS), s_kt = smem_u32(smem + S::KT),
                 s_bmt = smem_u32(smem + S::BMT), s_kh = smem_u32(smem + S::KH), s_tbt = smem_u32(smem + S::TBT),
                 s_v = smem_u32(smem + S::V), s_do = smem_u32(smem + S::DO), s_id = smem_u32(smem + S::ID);
  // K-major operand: k-step ks of 16 inside blocks of 64 (block stride bstride)
  auto kmaj = [](uint32_t base, int ks, uint32_t bstride) {
    return tc::desc_sw128(base + (uint32_t)(ks >> 2) * bstride + 32u * (uint32_t)(ks & 3));
  };
  // MN-major operand: k-step ks of 16 = two 1024-byte K atoms; lbo = stride between 64-element atoms
  auto mnmaj = [](uint32_t base, int ks, uint32_t lbo) { return tc::desc_sw128_mn(base + 2048u * (uint32_t)ks, lbo); };

  // ---------------------------------------------------------------- group A
  if (tid == 0) {
    // -V'^T [v][tok] = V^T (-I) + S^T Kt^T
    for (int ks = 0; ks < 4; ++ks)
      tc::mma_bf16(tmem + T_VP, mnmaj(s_v, ks, 8192), kmaj(s_id, ks, 0), tc::idesc_bf16_mn(128, 64, true, false), ks > 0);
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_VP, kmaj(s_ss, ks, 16384), kmaj(s_kt, ks, 8192), tc::idesc_bf16(128, 64), 1);
    // dU^T [v][r] = dO^T Bm + dS^T Kh^T
    for (int ks = 0; ks < 4; ++ks)
      tc::mma_bf16(tmem + T_DU, mnmaj(s_do, ks, 8192), kmaj(s_bmt, ks, 0), tc::idesc_bf16_mn(128, 64, true, false), ks > 0);
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_DU, kmaj(s_sds, ks, 16384), kmaj(s_kh, ks, 8192), tc::idesc_bf16(128, 64), 1);
    // dQt^T [k][r] = S dO^T: A = S (k rows) MN-major over S^T, B = dO [r][v] K-major
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_DQ, mnmaj(s_ss, ks, 16384), kmaj(s_do, ks, 8192), tc::idesc_bf16_mn(128, 64, true, false), ks > 0);
    tc::commit(&bar[1]);
  }
  // dgC_c = sum_v S^T[v][c] dS^T[v][c] while group A runs (two threads per channel)
  {
    const TileSW<128> sS((bf16 *)(smem + S::SS)), sdS((bf16 *)(smem + S::SDS));
    const int c = tid & 127, half = tid >> 7;
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int vv = 64 * half; vv < 64 * half + 64; vv += 4)
#pragma unroll
      for (int u = 0; u < 4; ++u) s4[u] = fmaf(to_f(*sS.at(vv + u, c)), to_f(*sdS.at(vv + u, c)), s4[u]);
    float *xch = reinterpret_cast<float *>(smem + S::XCH);
    if (half) xch[c] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    __syncthreads();
    if (!half) reinterpret_cast<float *>(rec + GradLayout::dgc)[c] = (s4[0] + s4[1]) + (s4[2] + s4[3]) + xch[c];
  }
  ok = mbar_wait(&bar[1], 0);
  tc::fence_after();
  // E: 32 columns of a [channel][tok] accumulator -> bf16 operand tile rows = channel (K-major over tok)
  auto to_tile = [&](uint32_t col, uint32_t tile_off, float sign) {
    float v[32];
    ld32(tl + col + 32 * hf, v);
    tc::wait_ld();
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = sign * v[8 * cb + i];
      *reinterpret_cast<uint4 *>(smem + tile_off + tc::sw128_off(128, row, 32 * hf + 8 * cb)) = tc::pack8(x);
    }
  };
  // E: 32 columns (r) of a [k][r] accumulator -> bf16 [r][k] rows of the gradient record, through this
  // warp's 32 x 32 block of the staging tile (rows 32 hf.., columns 32 qw..), 16-byte stores
  auto to_record = [&](uint32_t col, size_t rec_off, float sign) {
    float v[32];
    ld32(tl + col + 32 * hf, v);
    tc::wait_ld();
    bf16 *stg = reinterpret_cast<bf16 *>(smem + S::STG);
#pragma unroll
    for (int i = 0; i < 32; ++i) stg[(32 * hf + i) * 128 + row] = __float2bfloat16_rn(sign * v[i]);
    __syncwarp();
    bf16 *dst = reinterpret_cast<bf16 *>(rec + rec_off);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = 32 * hf + 8 * k + (lane >> 2), c8 = 32 * qw + 8 * (lane & 3);
      *reinterpret_cast<uint4 *>(dst + r * 128 + c8) = *reinterpret_cast<const uint4 *>(stg + r * 128 + c8);
    }
    __syncwarp();
  };
  if (ok) {
    to_tile(T_VP, S::VPT, -1.f);   // V'^T (over the dead Kt tile)
    to_tile(T_DU, S::DUT, 1.f);    // dU^T (over the dead V tile)
    to_record(T_DQ, GradLayout::dqt, 1.f);
  }
  fence_proxy_async();
  tc::fence_before();
  if (!__syncthreads_and(ok)) {
    report(p.status, ERR_TIMEOUT);
    if (warp == 0) tc::dealloc(tmem, 512);
    return;
  }
  tc::fence_after();

  // ---------------------------------------------------------------- group B
  const uint32_t s_vpt = smem_u32(smem + S::VPT), s_dut = smem_u32(smem + S::DUT);
  if (tid == 0) {
    // U^T [v][r] = V'^T Tb^T: B(n = r, k = j) = Tb[r][j] = Tb^T tile[j][r] -> MN-major
    for (int ks = 0; ks < 4; ++ks)
      tc::mma_bf16(tmem + T_U, kmaj(s_vpt, ks, 0), mnmaj(s_tbt, ks, 8192), tc::idesc_bf16_mn(128, 64, false, true), ks > 0);
    // dV'^T [v][j] = dU^T Tb: B(n = j, k = r) = Tb[r][j] = Tb^T tile[j][r] -> K-major
    for (int ks = 0; ks < 4; ++ks)
      tc::mma_bf16(tmem + T_DV, kmaj(s_dut, ks, 0), kmaj(s_tbt, ks, 0), tc::idesc_bf16(128, 64), ks > 0);
    // dTb [r][j] = dU V'^T (M = 64): A(m = r, k = v) = dU^T tile[v][r], B(n = j, k = v) = V'^T tile[v][j]
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_DTB, mnmaj(s_dut, ks, 8192), mnmaj(s_vpt, ks, 8192), tc::idesc_bf16_mn(64, 64, true, true), ks > 0);
    tc::commit(&bar[2]);
  }
  ok = mbar_wait(&bar[2], 0);
  tc::fence_after();
  // E: 32 columns (j) of an M = 64 accumulator row r -> masked (j <= r) row of the gradient record
  const int r64 = 16 * qw + (lane & 15);   // row of this lane in an M = 64 accumulator (lanes < 16)
  if (ok) {
    to_tile(T_U, S::UT, 1.f);     // U^T (the V'^T tile is done)
    to_tile(T_DV, S::DVT, 1.f);   // dV'^T (the dU^T tile is done)
    float v[32];
    ld32(tl + T_DTB + 32 * hf, v);
    tc::wait_ld();
    if (lane < 16) {
      float *dtb = reinterpret_cast<float *>(rec + GradLayout::dtb) + r64 * 64 + 32 * hf;
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = (32 * hf + 4 * c4 + e <= r64) ? v[4 * c4 + e] : 0.f;
        *reinterpret_cast<float4 *>(dtb + 4 * c4) = make_float4(x[0], x[1], x[2], x[3]);
      }
    }
  }
  fence_proxy_async();
  tc::fence_before();
  if (!__syncthreads_and(ok)) {
    report(p.status, ERR_TIMEOUT);
    if (warp == 0) tc::dealloc(tmem, 512);
    return;
  }
  tc::fence_after();

  // ---------------------------------------------------------------- group C
  const uint32_t s_ut = smem_u32(smem + S::UT), s_dvt = smem_u32(smem + S::DVT);
  if (tid == 0) {
    // dBm [r][j] = dO U^T (M = 64): A = dO [r][v] K-major, B(n = j, k = v) = U^T tile[v][j] MN-major
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_DBM, kmaj(s_do, ks, 8192), mnmaj(s_ut, ks, 8192), tc::idesc_bf16_mn(64, 64, false, true), ks > 0);
    // dKh^T [k][r] = dS U^T: A = dS (k rows) MN-major over dS^T, B(n = r, k = v) = U^T tile[v][r] MN-major
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_DKH, mnmaj(s_sds, ks, 16384), mnmaj(s_ut, ks, 8192), tc::idesc_bf16_mn(128, 64, true, true), ks > 0);
    // dV' S^T transposed: [k][r] = S dV'^T (negated in the epilogue: dKt = -dV' S^T)
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_DKT, mnmaj(s_ss, ks, 16384), mnmaj(s_dvt, ks, 8192), tc::idesc_bf16_mn(128, 64, true, true), ks > 0);
    tc::commit(&bar[3]);
  }
  ok = mbar_wait(&bar[3], 0);
  tc::fence_after();
  if (ok) {
    float v[32];
    ld32(tl + T_DBM + 32 * hf, v);
    tc::wait_ld();
    if (lane < 16) {
      bf16 *dbm = reinterpret_cast<bf16 *>(rec + GradLayout::dbm) + r64 * 64 + 32 * hf;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = (32 * hf + 8 * cb + e <= r64) ? v[8 * cb + e] : 0.f;
        *reinterpret_cast<uint4 *>(dbm + 8 * cb) = tc::pack8(x);
      }
    }
    to_record(T_DKH, GradLayout::dkh, 1.f);
    to_record(T_DKT, GradLayout::dkt, -1.f);
  } else {
    report(p.status, ERR_TIMEOUT);
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, 512);
}

cudaError_t launch_bwd_state_tc(const BwdStateParams &p, cudaStream_t s) {
  if (p.geo.max_chunks == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       St5Smem::BYTES);
  if (e != cudaSuccess) return e;
  kda_bwd_state_tc_kernel<<<dim3(p.geo.max_chunks, p.geo.heads), ST5_THREADS, St5Smem::BYTES, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
