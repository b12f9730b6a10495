// kda_bwd_tc.cu -- chunk-parallel part of the KDA backward on 5th-generation tensor cores.
//
// The reverse dS scan (kda_scan_tc.cu) leaves, for every chunk, the state gradient dS
// at the chunk end and the value gradient dv. One kernel then finishes all chunk-local
// gradients of a (chunk, head): one CTA of 8 warps, one CTA per SM.
//
// State side, with S the chunk-start state (forward) and dS the chunk-end state
// gradient, both kept as S^T [v][k] tiles:
//   V' = V - Kt S,   U = Tb V',   dU = Bm^T dO + Kh dS,   dV' = Tb^T dU
//   dQt = dO S^T,   dKt = -dV' S^T,   dKh = U dS^T,
//   dBm = dO U^T (j <= r),   dTb = dU V'^T (j <= r),   dgC_c = sum_v S_cv dS_cv
// and, through Tb = T Diag(beta) and T = (I + Diag(beta) A)^-1 (A, T from the prep):
//   dT = dTb Diag(beta),  X = dT T^T,  dL = -T^T X (strict lower),  dA = Diag(beta) dL,
//   dbeta_j = sum_r dTb_rj T_rj + sum_i dL_ji A_ji   (beta enters only through T and Tb).
// Every product is a tcgen05 MMA whose operands are tiles already in shared memory,
// read K-major or MN-major as each product needs (a tile of rows x 128 bytes in the
// 128-byte swizzle is K-major for one orientation and MN-major for the other). X and
// dL are kind::tf32 products of fp32 tiles (T, dT, X^T, T^T): the 64 x 64 products
// through T need more than bf16 precision.
//
// Intra-chunk side, through the bounded gating factors of the prep (kda_prep.cu): for
// r in sub-block a, x_r = e^{G_r-E_{a-1}}, y_r = e^{E_a-G_r}, the factor tiles
//   QL = q^ x,  KL = k^ x,  R = k^ y,  with Qt = QL P_a, Kt = KL P_a, Kh = R F_a,
// Bm = blocks of QL (R o D_ab)^T, A = blocks of KL (R o D_ab)^T (P_a = e^{E_{a-1}},
// F_a = e^{E_3-E_a}, D_ab = e^{E_{a-1}-E_b}). Their gradients, channel-major (TMEM
// lane = channel c), for r in sub-block t:
//   dQL = sum_{b<=t} D_tb o (R_b^T dBm_tb^T) + dQt P_t
//   dKL = sum_{b<=t} D_tb o (R_b^T dA_tb^T)  + dKt P_t
//   dR  = sum_{a>=t} D_at o (QL_a^T dBm_at + KL_a^T dA_at) + dKh F_t
// (M = 128 channels, N = K = 16 MMAs), then dq^ = dQL x, dk^ = dKL x + dR y,
// dG = dQL QL + dKL KL - dR R, dg = reverse cumulative sum of dG inside the chunk
// plus e^{G_last} (dgC + sum_r dKh_r Kh_r), and the L2-norm backward gives dq, dk.
// dQt, dKt and dKh never leave tensor memory. The diagonal of Bm, Bm_rr = q^_r . k^_r,
// does not depend on the gates: it is left out of the factor products (whose two
// contributions to dG_r would cancel only up to the rounding of the bf16 factor tiles,
// an error that does not shrink with dg under strong decay) and enters dq^ and dk^
// directly as dBm_rr k^_r and dBm_rr q^_r.
//
// Waits are bounded; on a timeout the CTA reports KDA_ERR_TIMEOUT, frees its tensor
// memory and returns.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc05.cuh"

namespace kda {

constexpr int BC_THREADS = 256;

struct BcSmem {
  static constexpr int SS = 0, SDS = 32768;            // S^T, dS^T [v][k] bf16, K-major over k (2 blocks of 16 KB)
  static constexpr int KT = 65536;                     // Kt [tok][k] bf16 (2 blocks of 8 KB)
  static constexpr int KHT = 81920, BM = KHT + 16384;  // the record's B2 tile: Kh^T [k][tok] and Bm [r][j]
  static constexpr int TB = 106496;                    // the record's Tb [r][j] (+ e^{G_last}, unused here)
  static constexpr int V = 115712;                     // V [tok][v] bf16, plain 256-byte rows
  static constexpr int DO = 132096;                    // dO [tok][v] bf16, K-major over v (2 blocks of 8 KB)
  static constexpr int BAR = 148480, TSLOT = BAR + 128;
  static constexpr int TK = 149504;                    // T [m][j], then T^T [r][m]: fp32 K-major (2 blocks of 8 KB)
  static constexpr int QR = TK + 16384, KR = QR + 16384;   // raw q, k [64][128] bf16 rows
  static constexpr int MISC = KR + 16384;
  static constexpr int RQ0 = MISC, RK = RQ0 + 256;     // [64] inverse row norms of q, k
  static constexpr int TOT = RK + 256;                 // [4][128] sub-block gate sums (log2 units)
  static constexpr int PV = TOT + 2048, FV = PV + 2048;   // [4][128] P_a, F_a
  static constexpr int DV = FV + 2048;                 // [10][128] D_ab, pair a(a+1)/2 + b
  static constexpr int TAIL = DV + 5120;               // [128] dgC e^{G_last}
  static constexpr int CSUM = TAIL + 512;              // [2][128] halves of sum_r dKh_rc Kh_rc
  static constexpr int XS = CSUM + 1024;               // [2][128] half-block sums of dG
  static constexpr int RD = XS + 1024;                 // [2][4][16] partial row dots
  static constexpr int DB1P = RD + 512, DB2P = DB1P + 1024, SB = DB2P + 512;
  static constexpr int DBD = SB + 256;                 // [64] diagonal of dBm (fp32)
  static constexpr int DGCP = DBD + 256;               // [16][128] partial row dots of S and dS
  static constexpr int END = DGCP + 8192;
  static constexpr int BYTES = END + 1024;             // + alignment slack
  // regions reused once their first contents are consumed
  static constexpr int VPT = KT, UT = KT;              // V'^T, then U^T [v][tok] (groups A, B)
  static constexpr int DUT = V, DVT = V;               // dU^T, then dV'^T [v][tok]
  static constexpr int DT0 = TB, DT1 = BM;             // dT [r][j] fp32 K-major: the two 8 KB K-blocks (group C)
  static constexpr int XT = SS;                        // X^T [j][m] fp32 K-major (group D)
  static constexpr int AS = DO;                        // A fp32 [64][64] in the layout of T (group D)
  static constexpr int CSA = SS + 16384, CSB = KHT;    // local gate sums (log2) of rows 0..31, 32..63: [32][128] fp32
  static constexpr int DBM = BM;                       // dBm [r][j] bf16 (rounds; read K-major and MN-major)
  static constexpr int DA = V;                         // dA [r][j] bf16 (rounds; read K-major and MN-major)
  static constexpr int QLF = SDS, KLF = SDS + 16384, RF = KT;   // factor tiles [r][c] bf16 (rounds)
};

namespace {
// TMEM columns (512 allocated). dKt^T, dQt^T, dKh^T (320..511) live until the end.
constexpr uint32_t T_VP = 0, T_DU = 64, T_U = 128, T_DV = 192, T_DTB = 256, T_DBM = 0, T_X = 64, T_DL = 128,
                   T_DKT = 320, T_DQ = 384, T_DKH = 448, T_R0 = 0, T_R1 = 144;

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

// 2^x by the hardware approximation (relative error about 2^-22), results below 2^-126 flushed to
// zero: every gating factor here is at most 1 and multiplies O(1) values. The round epilogues and
// the Kh sum both form their factors with it, so the two agree to the last bit.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Warp-collective: 8 consecutive fp32 columns of TMEM lane (lane base + thread).
__device__ __forceinline__ void ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// K-major operand: k-step ks of 16 bf16 (or 8 fp32) inside blocks of 64 bf16 (bstride apart)
__device__ __forceinline__ uint64_t kmaj(uint32_t base, int ks, uint32_t bstride) {
  return tc::desc_sw128(base + (uint32_t)(ks >> 2) * bstride + 32u * (uint32_t)(ks & 3));
}
// MN-major operand: k-step ks of 16 = two 1024-byte K atoms; lbo = stride between 64-element atoms
__device__ __forceinline__ uint64_t mnmaj(uint32_t base, int ks, uint32_t lbo) {
  return tc::desc_sw128_mn(base + 2048u * (uint32_t)ks, lbo);
}

struct RoundCtx {
  const BwdChunkParams *p;
  const ChunkRef *ref;
  char *smem;
  uint32_t tl;                // this warp's TMEM lane base
  int c, hf, qw, lane, h;
  float run;                  // dg suffix sum of the rows after the current block
};

// Epilogue of round t (rows 16t..16t+15): this thread has channel c and rows 16t + 8 hf + i.
// One copy of the code for all four rounds (t is a run-time value): the kernel is long and
// runs one CTA per SM, so its instruction footprint matters. `after_read` runs right after the
// CTA barrier that follows every thread's tensor-memory reads (it issues the round that reuses
// this buffer).
template <class AfterRead>
__device__ __forceinline__ void round_epilogue(RoundCtx &x, const int t, uint32_t base, AfterRead after_read) {
  using S = BcSmem;
  const BwdChunkParams &p = *x.p;
  const int c = x.c, hf = x.hf;
  // shared memory: local gate sums, raw q, k of this thread's rows
  float csv[8], qv[8], kv[8];
  const bf16 *sq_ = (const bf16 *)(x.smem + S::QR), *sk_ = (const bf16 *)(x.smem + S::KR);
  const float *csb = (const float *)(x.smem + (t < 2 ? S::CSA : S::CSB)) + (16 * (t & 1) + 8 * hf) * 128 + c;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 16 * t + 8 * hf + i;
    csv[i] = csb[i * 128];
    qv[i] = to_f(sq_[r * D + c]);
    kv[i] = to_f(sk_[r * D + c]);
  }
  const float(*tot)[128] = (const float(*)[128])(x.smem + S::TOT);
  const float(*pv)[128] = (const float(*)[128])(x.smem + S::PV);
  const float(*fv)[128] = (const float(*)[128])(x.smem + S::FV);
  const float(*dvp)[128] = (const float(*)[128])(x.smem + S::DV);
  const float *rq0 = (const float *)(x.smem + S::RQ0), *rk = (const float *)(x.smem + S::RK);
  const float *dbd = (const float *)(x.smem + S::DBD);
  const float pa = pv[t][c], fa = fv[t][c], tt = tot[t][c];
  // tensor memory: the round's pair products (t + 6 blocks of 8 columns for this thread) and
  // dQt^T, dKt^T, dKh^T, issued together (warp-uniform predicates) with one wait
  float pp[NSUB][8], pq[NSUB][8], pw[NSUB][8], gq[8], gk[8], gh[8];
  ld8(x.tl + T_DQ + 16 * t + 8 * hf, gq);
  ld8(x.tl + T_DKT + 16 * t + 8 * hf, gk);   // holds -dKt^T
  ld8(x.tl + T_DKH + 16 * t + 8 * hf, gh);
#pragma unroll
  for (int b = 0; b < NSUB; ++b)
    if (b <= t) {
      ld8(x.tl + base + 16 * b + 8 * hf, pp[b]);
      ld8(x.tl + base + 16 * (t + 1) + 16 * b + 8 * hf, pq[b]);
    }
#pragma unroll
  for (int aa = 0; aa < NSUB; ++aa)
    if (aa >= t) ld8(x.tl + base + 32 * (t + 1) + 16 * (aa - t) + 8 * hf, pw[aa]);
  tc::wait_ld();
  // pair products scaled by the pair factors as they are summed
  float tq[8], tk[8], tw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) tq[i] = tk[i] = tw[i] = 0.f;
#pragma unroll
  for (int b = 0; b < NSUB; ++b)
    if (b <= t) {
      const float d = dvp[t * (t + 1) / 2 + b][c];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        tq[i] = fmaf(d, pp[b][i], tq[i]);
        tk[i] = fmaf(d, pq[b][i], tk[i]);
      }
    }
#pragma unroll
  for (int aa = 0; aa < NSUB; ++aa)
    if (aa >= t) {
      const float d = dvp[aa * (aa + 1) / 2 + t][c];
#pragma unroll
      for (int i = 0; i < 8; ++i) tw[i] = fmaf(d, pw[aa][i], tw[i]);
    }
  // per row: factor values in fp32, factor-tile gradients, dq^, dk^, dG
  const int len = x.ref->len;
  const long long t0 = x.ref->t0;
  const int H = p.geo.heads;
  float dq_[8], dk_[8], dG[8], rv[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 16 * t + 8 * hf + i;
    const float xx = ex2(csv[i]), yy = ex2(tt - csv[i]);
    const float qh = qv[i] * rq0[r], kh = kv[i] * rk[r];
    const float ql = p.scale * qh * xx, kl = kh * xx, rr = kh * yy;
    const float dQL = fmaf(gq[i], pa, tq[i]), dKL = fmaf(-gk[i], pa, tk[i]), dR = fmaf(gh[i], fa, tw[i]);
    const float bd = dbd[r];   // dBm_rr: Bm_rr = (scale q^_r) . k^_r
    dq_[i] = fmaf(bd, kh, dQL * xx);
    dk_[i] = fmaf(dKL, xx, fmaf(dR, yy, bd * p.scale * qh));
    dG[i] = fmaf(dQL, ql, fmaf(dKL, kl, -dR * rr));   // natural-log units
    rv[i] = qh * dq_[i];
    rv[8 + i] = kh * dk_[i];
  }
  // row dots over the 128 channels: recursive halving across the warp (value index
  // 8 b4 + 4 b3 + 2 b2 + b1 of the lane ends up in lane pairs), then the 4 warps of this
  // column half through shared memory
  const int lane = x.lane;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool up = lane & 16;
    const float send = up ? rv[i] : rv[i + 8], keep = up ? rv[i + 8] : rv[i];
    rv[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool up = lane & 8;
    const float send = up ? rv[i] : rv[i + 4], keep = up ? rv[i + 4] : rv[i];
    rv[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool up = lane & 4;
    const float send = up ? rv[i] : rv[i + 2], keep = up ? rv[i + 2] : rv[i];
    rv[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  {
    const bool up = lane & 2;
    const float send = up ? rv[0] : rv[1], keep = up ? rv[1] : rv[0];
    rv[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  rv[0] += __shfl_xor_sync(0xffffffffu, rv[0], 1);
  float *rd = (float *)(x.smem + S::RD) + hf * 64;
  if (!(lane & 1)) {
    const int idx = 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
    rd[x.qw * 16 + idx] = rv[0];
  }
  named_sync(1 + hf, 128);
  float *xs = (float *)(x.smem + S::XS);
  float sdg = 0.f;
  float dq4[8], dk4[8];   // the 4 warps' partial row dots, 16-byte reads
#pragma unroll
  for (int hlf = 0; hlf < 2; ++hlf) {
    float4 sq4 = make_float4(0.f, 0.f, 0.f, 0.f), sk4 = sq4;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float4 a4 = *reinterpret_cast<const float4 *>(rd + 16 * w + 4 * hlf);
      const float4 b4 = *reinterpret_cast<const float4 *>(rd + 16 * w + 8 + 4 * hlf);
      sq4.x += a4.x; sq4.y += a4.y; sq4.z += a4.z; sq4.w += a4.w;
      sk4.x += b4.x; sk4.y += b4.y; sk4.z += b4.z; sk4.w += b4.w;
    }
    dq4[4 * hlf] = sq4.x; dq4[4 * hlf + 1] = sq4.y; dq4[4 * hlf + 2] = sq4.z; dq4[4 * hlf + 3] = sq4.w;
    dk4[4 * hlf] = sk4.x; dk4[4 * hlf + 1] = sk4.y; dk4[4 * hlf + 2] = sk4.z; dk4[4 * hlf + 3] = sk4.w;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 16 * t + 8 * hf + i;
    const float dotq = dq4[i], dotk = dk4[i];
    if (r < len) {
      const size_t off = ((size_t)(t0 + r) * H + x.h) * D + c;
      const float r0 = rq0[r], rkr = rk[r];
      p.dq[off] = p.scale * r0 * (dq_[i] - qv[i] * r0 * dotq);
      p.dk[off] = rkr * (dk_[i] - kv[i] * rkr * dotk);
    }
    sdg += dG[i];
  }
  xs[hf * 128 + c] = sdg;
  tc::fence_before();
  __syncthreads();   // the half sums are in place and every thread's reads of this buffer are done
  tc::fence_after();
  after_read();
  const float other = xs[(1 - hf) * 128 + c];
  float acc = x.run + (hf ? 0.f : other);
#pragma unroll
  for (int i = 7; i >= 0; --i) {
    const int r = 16 * t + 8 * hf + i;
    acc += dG[i];
    if (r < len) p.dg[((size_t)(t0 + r) * H + x.h) * D + c] = acc;
  }
  x.run += sdg + other;
}
}  // namespace

__global__ void __launch_bounds__(BC_THREADS, 1) kda_bwd_chunk_tc_kernel(const __grid_constant__ BwdChunkParams p) {
  using S = BcSmem;
  extern __shared__ __align__(1024) char smem_raw[];
  char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int H = p.geo.heads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qw = warp & 3, hf = warp >> 2;          // lane quarter, column half
  const int row = 32 * qw + lane;                   // TMEM lane of this thread
  const int r64 = 16 * qw + (lane & 15);            // row of this lane in an M = 64 accumulator (lanes < 16)
  // [0] loads, [1..4] groups A-D, [5..8] rounds, [9] A, [10] the next block's prefetched tiles
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::BAR);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + S::TSLOT);
  float *sb = reinterpret_cast<float *>(smem + S::SB);
  float *rq0 = reinterpret_cast<float *>(smem + S::RQ0), *rk = reinterpret_cast<float *>(smem + S::RK);
  float(*tot)[128] = (float(*)[128])(smem + S::TOT);
  float(*pv)[128] = (float(*)[128])(smem + S::PV);
  float(*fv)[128] = (float(*)[128])(smem + S::FV);
  float(*dvp)[128] = (float(*)[128])(smem + S::DV);

  if (tid == 0) {
    // groups A-C and the rounds are issued by two threads (one commit each), the rest by one
    for (int i = 0; i < 11; ++i) mbar_init(&bar[i], (i >= 1 && i <= 3) || (i >= 5 && i <= 8) ? 2 : 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tl = tmem + ((uint32_t)(32 * qw) << 16);
  auto fail_out = [&]() {
    report(p.status, ERR_TIMEOUT);
    if (warp == 0) tc::dealloc(tmem, 512);
  };

  // Persistent: CTA b runs blocks b, b + grid, ... in head-fastest order (the CTAs resident at
  // one time cover whole token rows [t][all heads][d] and consecutive chunk records). While a
  // block's round epilogues run, the next block's dO, T and first S^T block are fetched into
  // the tiles the rounds no longer use.
  const long long nblk = (long long)p.geo.max_chunks * H;
  // the chunk of the block this CTA runs next is looked up one block ahead (during the
  // current block's products), so a block starts with its loads
  ChunkRef cur;
  bool have_cur = blockIdx.x < nblk && chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, (int)(blockIdx.x / H), cur);
  int it = 0;
  for (long long blk = blockIdx.x; have_cur; blk += gridDim.x, ++it) {
  const int h = (int)(blk % H), chunk = (int)(blk / H);
  const ChunkRef ref = cur;
  const uint32_t ph = (uint32_t)(it & 1);
  const bool pre = it > 0;   // the previous block prefetched this block's dO, T, S^T block 0 and Tb
  const long long nb = blk + gridDim.x;   // the block this CTA runs next, if any
  const int nh = (int)(nb % H);
  const size_t nrid = (size_t)(nb / H) * H + nh;
  const size_t rid = (size_t)chunk * H + h;

  // ---------------------------------------------------------------- loads
  // Thread 0 issues the block's copies first; every thread then loads its gate rows (thread =
  // channel pair x sub-block, plain loads into registers) and this token's beta, whose latency
  // overlaps the copies. (The plain loads queue behind the previous block's gradient stores, so
  // issuing them before the copies would hold the copies back.)
  // bulk copies of the saved tiles and the record; TMA boxes of this chunk's V, dO, q, k rows
  // (rows past the tensor read as zero) and of T
  const int t0i = (int)ref.t0, arow = (int)rid * 128;
  if (tid == 0) {
    const char *rb = (const char *)p.img + rid * TcRec::BYTES;
    fence_proxy_async();
    mbar_expect_tx(&bar[0], (pre ? 16384 : 32768) + 32768 + (TcRec::TB - TcRec::B2) + (pre ? 0 : TcRec::BYTES - TcRec::TB) +
                                KtRec::BYTES + (pre ? 3 : 5) * 16384);
    if (pre)
      bulk_g2s(smem + S::SS + 16384, (const char *)p.saved + rid * 32768 + 16384, 16384, &bar[0]);
    else
      bulk_g2s(smem + S::SS, (const char *)p.saved + rid * 32768, 32768, &bar[0]);
    bulk_g2s(smem + S::SDS, (const char *)p.dsaved + rid * 32768, 32768, &bar[0]);
    bulk_g2s(smem + S::KHT, rb + TcRec::B2, TcRec::TB - TcRec::B2, &bar[0]);        // Kh^T, Bm
    if (!pre) bulk_g2s(smem + S::TB, rb + TcRec::TB, TcRec::BYTES - TcRec::TB, &bar[0]);   // Tb, e^{G_last}
    bulk_g2s(smem + S::KT, (const char *)p.kt + rid * KtRec::BYTES, KtRec::BYTES, &bar[0]);   // Kt
    tc::tma_load_3d(smem + S::V, &p.tm_v, 0, h, t0i, &bar[0]);
    if (!pre) {
      tc::tma_load_3d(smem + S::DO, &p.tm_do, 0, h, t0i, &bar[0]);
      tc::tma_load_3d(smem + S::DO + 8192, &p.tm_do, 64, h, t0i, &bar[0]);
    }
    tc::tma_load_3d(smem + S::QR, &p.tm_q, 0, h, t0i, &bar[0]);
    tc::tma_load_3d(smem + S::KR, &p.tm_k, 0, h, t0i, &bar[0]);
    if (!pre) {
      tc::tma_load_2d(smem + S::TK, &p.tm_aux, 0, arow + 64, &bar[0]);
      tc::tma_load_2d(smem + S::TK + 8192, &p.tm_aux, 32, arow + 64, &bar[0]);
    }
  }
  const int cp = tid & 63, a = tid >> 6, c0 = 2 * cp;
  float2 csr[SUB];
#pragma unroll
  for (int i = 0; i < SUB; ++i) {
    const int rr = a * SUB + i;
    csr[i] = rr < ref.len ? *reinterpret_cast<const float2 *>(p.g + ((size_t)(ref.t0 + rr) * H + h) * D + c0)
                          : make_float2(0.f, 0.f);
  }
  const float beta_t = tid < 64 && tid < ref.len ? p.beta[(size_t)(ref.t0 + tid) * H + h] : 0.f;
  // while the copies land: the gate scan; the local sums G_r - E_{a-1} (log2) stay in registers
  // for the factor tiles
  {
    float2 run = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < SUB; ++i) {
      run.x = fmaf(csr[i].x, LOG2E, run.x);
      run.y = fmaf(csr[i].y, LOG2E, run.y);
      csr[i] = run;
    }
    tot[a][c0] = run.x;
    tot[a][c0 + 1] = run.y;
  }
  if (tid < 64) sb[tid] = beta_t;
  bool ok = mbar_wait(&bar[0], ph);
  if (pre) ok &= mbar_wait(&bar[10], (uint32_t)((it - 1) & 1));
  if (ref.len < CH && ok) {
    // a sequence's last chunk: rows past its end read as zero (the boxes hold the next sequence's rows)
    for (int idx = tid; idx < (CH - ref.len) * 16; idx += BC_THREADS) {
      const int r = ref.len + (idx >> 4), ch = idx & 15;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4 *>(smem + S::V + r * 256 + 16 * ch) = z;
      *reinterpret_cast<uint4 *>(smem + S::QR + r * 256 + 16 * ch) = z;
      *reinterpret_cast<uint4 *>(smem + S::KR + r * 256 + 16 * ch) = z;
      *reinterpret_cast<uint4 *>(smem + S::DO + (ch >> 3) * 8192 + r * 128 + 16 * (ch & 7)) = z;
    }
    fence_proxy_async();
  }
  tc::fence_before();
  if (!__syncthreads_and(ok)) return fail_out();
  tc::fence_after();

  const uint32_t s_ss = smem_u32(smem + S::SS), s_sds = smem_u32(smem + S::SDS), s_kt = smem_u32(smem + S::KT),
                 s_bm = smem_u32(smem + S::BM), s_kht = smem_u32(smem + S::KHT), s_tb = smem_u32(smem + S::TB),
                 s_do = smem_u32(smem + S::DO);

  // ---------------------------------------------------------------- group A
  // Every MMA costs its issuing thread about 50 cycles whatever its size, so each group's
  // independent accumulator chains are split between two threads in different warps (0 and 32),
  // each committing once to the group's barrier (two arrivals).
  if (tid == 0) {
    // (Kt S)^T [v][j] = S^T Kt^T; V'^T = V^T - (Kt S)^T in the epilogue
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_VP, kmaj(s_ss, ks, 16384), kmaj(s_kt, ks, 8192), tc::idesc_bf16(128, 64), ks > 0);
    // dQt^T [k][r] = S dO^T: A = S (k rows) MN-major over S^T, B = dO [r][v] K-major
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_DQ, mnmaj(s_ss, ks, 16384), kmaj(s_do, ks, 8192), tc::idesc_bf16_mn(128, 64, true, false), ks > 0);
    tc::commit(&bar[1]);
  } else if (tid == 32) {
    // dU^T [v][j] = dO^T Bm + dS^T Kh^T: B(n = j, k = r) = Bm[r][j] and B(n = j, k = dk) = Kh^T[dk][j],
    // both rows k of the record's tiles -> MN-major
    for (int ks = 0; ks < 4; ++ks)
      tc::mma_bf16(tmem + T_DU, mnmaj(s_do, ks, 8192), mnmaj(s_bm, ks, 8192), tc::idesc_bf16_mn(128, 64, true, true), ks > 0);
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_DU, kmaj(s_sds, ks, 16384), mnmaj(s_kht, ks, 8192), tc::idesc_bf16_mn(128, 64, false, true), 1);
    tc::commit(&bar[1]);
  }
  ChunkRef nr;
  const bool have_next = nb < nblk && chunk_lookup(p.geo.chunk_off, p.geo.cu, p.geo.n_seqs, (int)(nb / H), nr);
  {
    // gate factors: E_{a-1}, E_3 per channel; pair factors D_ab, P_a, F_a
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
        dvp[pr][c0] = exp2f(em[0] - eb[0]);
        dvp[pr][c0 + 1] = exp2f(em[1] - eb[1]);
      }
    }
    pv[a][c0] = exp2f(em[0]);
    pv[a][c0 + 1] = exp2f(em[1]);
    fv[a][c0] = exp2f(e3[0] - em[0] - tot[a][c0]);
    fv[a][c0 + 1] = exp2f(e3[1] - em[1] - tot[a][c0 + 1]);
  }
  // row norms of q, k (4 threads per row, 32 channels each; the word order is rotated by row
  // so that the 8 rows of a warp read different banks)
  {
    const int r = tid >> 2, part = tid & 3, rot = 2 * (r & 7);
    const bf16 *sq_ = (const bf16 *)(smem + S::QR), *sk_ = (const bf16 *)(smem + S::KR);
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
      rq0[r] = rsqrtf(sq + 1e-6f);
      rk[r] = rsqrtf(sk + 1e-6f);
    }
  }
  // dgC_c e^{G_last}, dgC_c = sum_v S_cv dS_cv: 16-byte chunks (8 channels) of the S^T and dS^T
  // tiles, thread = (chunk j, 8 rows v), then the 16 row groups summed in a fixed order
  {
    const int j = tid & 15, vg = tid >> 4;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t o = tc::sw128_off(128, 8 * vg + i, 8 * j);
      const uint4 x = *reinterpret_cast<const uint4 *>(smem + S::SS + o);
      const uint4 y = *reinterpret_cast<const uint4 *>(smem + S::SDS + o);
      const uint32_t xv[4] = {x.x, x.y, x.z, x.w}, yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xv[e]));
        const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&yv[e]));
        acc[2 * e] = fmaf(fx.x, fy.x, acc[2 * e]);
        acc[2 * e + 1] = fmaf(fx.y, fy.y, acc[2 * e + 1]);
      }
    }
    float *part = reinterpret_cast<float *>(smem + S::DGCP);
    *reinterpret_cast<float4 *>(part + vg * 128 + 8 * j) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4 *>(part + vg * 128 + 8 * j + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    __syncthreads();
    if (tid < 128) {
      float sdg = 0.f;
#pragma unroll
      for (int g2 = 0; g2 < 16; ++g2) sdg += part[g2 * 128 + tid];
      const float e3 = (tot[0][tid] + tot[1][tid]) + (tot[2][tid] + tot[3][tid]);
      reinterpret_cast<float *>(smem + S::TAIL)[tid] = sdg * exp2f(e3);
    }
  }
  ok = __all_sync(0xffffffffu, mbar_wait(&bar[1], ph));
  tc::fence_after();
  // E: 32 columns of a [channel][tok] accumulator -> bf16 operand tile rows = channel (K-major over tok)
  auto to_tile = [&](uint32_t col, uint32_t tile_off) {
    float v[32];
    ld32(tl + col + 32 * hf, v);
    tc::wait_ld();
#pragma unroll
    for (int cb = 0; cb < 4; ++cb)
      *reinterpret_cast<uint4 *>(smem + tile_off + tc::sw128_off(128, row, 32 * hf + 8 * cb)) = tc::pack8(v + 8 * cb);
  };
  float du[32];
  if (ok) {
    // V'^T = V^T - (Kt S)^T over the dead Kt tile; dU^T is held until the V tile is done
    float v[32];
    ld32(tl + T_VP + 32 * hf, v);
    ld32(tl + T_DU + 32 * hf, du);
    tc::wait_ld();
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
      float x8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = 32 * hf + 8 * cb + i;
        x8[i] = to_f(*reinterpret_cast<const bf16 *>(smem + S::V + j * 256 + 2 * row)) - v[8 * cb + i];
      }
      *reinterpret_cast<uint4 *>(smem + S::VPT + tc::sw128_off(128, row, 32 * hf + 8 * cb)) = tc::pack8(x8);
    }
  }
  if (!__syncthreads_and(ok)) return fail_out();
#pragma unroll
  for (int cb = 0; cb < 4; ++cb)
    *reinterpret_cast<uint4 *>(smem + S::DUT + tc::sw128_off(128, row, 32 * hf + 8 * cb)) = tc::pack8(du + 8 * cb);
  fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  // ---------------------------------------------------------------- group B
  const uint32_t s_vpt = smem_u32(smem + S::VPT), s_dut = smem_u32(smem + S::DUT);
  if (tid == 0) {
    // U^T [v][r] = V'^T Tb^T: B(n = r, k = j) = Tb[r][j] -> K-major
    for (int ks = 0; ks < 4; ++ks)
      tc::mma_bf16(tmem + T_U, kmaj(s_vpt, ks, 0), kmaj(s_tb, ks, 0), tc::idesc_bf16(128, 64), ks > 0);
    // dV'^T [v][j] = dU^T Tb: B(n = j, k = r) = Tb[r][j] -> MN-major
    for (int ks = 0; ks < 4; ++ks)
      tc::mma_bf16(tmem + T_DV, kmaj(s_dut, ks, 0), mnmaj(s_tb, ks, 8192), tc::idesc_bf16_mn(128, 64, false, true), ks > 0);
    tc::commit(&bar[2]);
  } else if (tid == 32) {
    // dTb [r][j] = dU V'^T (M = 64): A(m = r, k = v) = dU^T tile[v][r], B(n = j, k = v) = V'^T tile[v][j]
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_DTB, mnmaj(s_dut, ks, 8192), mnmaj(s_vpt, ks, 8192), tc::idesc_bf16_mn(64, 64, true, true), ks > 0);
    tc::commit(&bar[2]);
  }
  ok = __all_sync(0xffffffffu, mbar_wait(&bar[2], ph));
  tc::fence_after();
  if (ok) {
    to_tile(T_U, S::UT);     // U^T (the V'^T tile is done)
    to_tile(T_DV, S::DVT);   // dV'^T (the dU^T tile is done)
    // dTb (masked j <= r) -> dT = dTb Diag(beta) as the fp32 K-major operand of X = dT T^T, and
    // the column sums sum_r dTb_rj T_rj (dbeta through Tb) by recursive halving over the 16 rows
    float v[32];
    ld32(tl + T_DTB + 32 * hf, v);
    tc::wait_ld();
    char *dtblk = smem + (hf ? S::DT1 : S::DT0);
    if (lane < 16) {
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const uint32_t o = (uint32_t)(r64 * 128 + (((c4 ^ (r64 & 7)) & 7) << 4));
        const float4 t4 = *reinterpret_cast<const float4 *>(smem + S::TK + hf * 8192 + o);
        float x4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) x4[e] = (32 * hf + 4 * c4 + e <= r64) ? v[4 * c4 + e] : 0.f;
        const int j = 32 * hf + 4 * c4;
        *reinterpret_cast<float4 *>(dtblk + o) =
            make_float4(x4[0] * sb[j], x4[1] * sb[j + 1], x4[2] * sb[j + 2], x4[3] * sb[j + 3]);
        v[4 * c4] = x4[0] * t4.x;
        v[4 * c4 + 1] = x4[1] * t4.y;
        v[4 * c4 + 2] = x4[2] * t4.z;
        v[4 * c4 + 3] = x4[3] * t4.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.f;
    }
    // after the step with offset o a lane keeps the half of its columns selected by (lane & o)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const bool up = lane & 8;
      const float send = up ? v[i] : v[i + 16], keep = up ? v[i + 16] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool up = lane & 4;
      const float send = up ? v[i] : v[i + 8], keep = up ? v[i + 8] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool up = lane & 2;
      const float send = up ? v[i] : v[i + 4], keep = up ? v[i + 4] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const bool up = lane & 1;
      const float send = up ? v[i] : v[i + 2], keep = up ? v[i + 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
    if (lane < 16) {
      const int col = 32 * hf + 16 * ((lane >> 3) & 1) + 8 * ((lane >> 2) & 1) + 4 * ((lane >> 1) & 1) + 2 * (lane & 1);
      float *db1 = reinterpret_cast<float *>(smem + S::DB1P) + qw * 64 + col;
      db1[0] = v[0];
      db1[1] = v[1];
    }
  }
  fence_proxy_async();
  tc::fence_before();
  if (!__syncthreads_and(ok)) return fail_out();
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
    tc::commit(&bar[3]);
  } else if (tid == 32) {
    // S dV'^T [k][r] = -dKt^T: A = S (k rows) MN-major over S^T, B(n = r, k = v) = dV'^T tile[v][r] MN-major
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_bf16(tmem + T_DKT, mnmaj(s_ss, ks, 16384), mnmaj(s_dvt, ks, 8192), tc::idesc_bf16_mn(128, 64, true, true), ks > 0);
    // X = dT T^T (tf32), formed transposed so each TMEM lane holds a row of the X^T operand tile:
    // X^T [m][r] = T dT^T, A = T [m][j], B = dT [r][j], both K-major (M = N = 64)
    const uint32_t s_dt = smem_u32(smem + S::DT0), s_tk = smem_u32(smem + S::TK);
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_tf32(tmem + T_X, kmaj(s_tk, ks, 8192), kmaj(s_dt, ks, (uint32_t)(S::DT1 - S::DT0)), tc::idesc_tf32(64, 64), ks > 0);
    tc::commit(&bar[3]);
  }
  ok = __all_sync(0xffffffffu, mbar_wait(&bar[3], ph));
  tc::fence_after();
  float tcol[16];   // T[m0 + e][r] for the in-place transpose of T (thread: r = tid % 64, m0 = 16 (tid / 64))
  if (ok) {
    // A of the prep into the dead dO tile, for the dbeta term of epilogue D
    if (tid == 0) {
      mbar_expect_tx(&bar[9], 16384);
      tc::tma_load_2d(smem + S::AS, &p.tm_aux, 0, arow, &bar[9]);
      tc::tma_load_2d(smem + S::AS + 8192, &p.tm_aux, 32, arow, &bar[9]);
    }
    {
      const int r = tid & 63, m0 = 16 * (tid >> 6);
#pragma unroll
      for (int e = 0; e < 16; ++e) tcol[e] = *reinterpret_cast<const float *>(smem + S::TK + tc::sw128_off32(64, m0 + e, r));
    }
    // dBm (strictly lower, j < r) -> bf16 dBm [r][j] and dBm^T [j][r] operand tiles (over the
    // dead dT blocks); its diagonal, in fp32, to DBD
    float v[32];
    ld32(tl + T_DBM + 32 * hf, v);
    tc::wait_ld();
    if (lane < 16) {
      float diag = 0.f;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        float x8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = 32 * hf + 8 * cb + e;
          x8[e] = j < r64 ? v[8 * cb + e] : 0.f;
          if (j == r64) diag = v[8 * cb + e];
        }
        *reinterpret_cast<uint4 *>(smem + S::DBM + tc::sw128_off(64, r64, 32 * hf + 8 * cb)) = tc::pack8(x8);
      }
      if ((r64 >> 5) == hf) reinterpret_cast<float *>(smem + S::DBD)[r64] = diag;
    }
    // X^T [j][m] (fp32 K-major over m) over the dead S^T tile, row by row
    ld32(tl + T_X + 32 * hf, v);
    tc::wait_ld();
    if (lane < 16) {
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        *reinterpret_cast<float4 *>(smem + S::XT + tc::sw128_off32(64, r64, 32 * hf + 4 * q4)) =
            make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
    }
  }
  if (!__syncthreads_and(ok)) return fail_out();
  {   // T^T [r][m] over T
    const int r = tid & 63, m0 = 16 * (tid >> 6);
#pragma unroll
    for (int e = 0; e < 16; e += 4)
      *reinterpret_cast<float4 *>(smem + S::TK + tc::sw128_off32(64, r, m0 + e)) =
          make_float4(tcol[e], tcol[e + 1], tcol[e + 2], tcol[e + 3]);
  }
  fence_proxy_async();
  tc::fence_before();
  __syncthreads();
  tc::fence_after();

  // ---------------------------------------------------------------- group D
  if (tid == 0) {
    // T^T X [r][j] (M = 64, tf32): A = T^T [r][m], B = X^T [j][m]; dL = -(T^T X)
    const uint32_t s_ttk = smem_u32(smem + S::TK), s_xt = smem_u32(smem + S::XT);
    for (int ks = 0; ks < 8; ++ks)
      tc::mma_tf32(tmem + T_DL, kmaj(s_ttk, ks, 8192), kmaj(s_xt, ks, 8192), tc::idesc_tf32(64, 64), ks > 0);
    tc::commit(&bar[4]);
  }
  // factor tiles QL, KL, R [r][c] (bf16, K-major over c) over the dead dS^T and U^T tiles, and the
  // local gate sums for the rounds: thread = channel pair x sub-block, as in the prep
  {
    const float ta0 = tot[a][c0], ta1 = tot[a][c0 + 1];
    const bf16 *sq_ = (const bf16 *)(smem + S::QR), *sk_ = (const bf16 *)(smem + S::KR);
#pragma unroll
    for (int i = 0; i < SUB; ++i) {
      const int r = a * SUB + i;
      const float2 run = csr[i];
      *reinterpret_cast<float2 *>(smem + (r < 32 ? S::CSA + r * 512 : S::CSB + (r - 32) * 512) + c0 * 4) = run;
      const float2 qf = ld2(sq_ + r * D + c0), kf = ld2(sk_ + r * D + c0);
      const float x0 = ex2(run.x), x1 = ex2(run.y), y0 = ex2(ta0 - run.x), y1 = ex2(ta1 - run.y);
      const float qs = p.scale * rq0[r], ks_ = rk[r];
      const uint32_t o = tc::sw128_off(64, r, c0);
      st2((bf16 *)(smem + S::QLF + o), qf.x * qs * x0, qf.y * qs * x1);
      st2((bf16 *)(smem + S::KLF + o), kf.x * ks_ * x0, kf.y * ks_ * x1);
      st2((bf16 *)(smem + S::RF + o), kf.x * ks_ * y0, kf.y * ks_ * y1);
    }
  }
  ok = __all_sync(0xffffffffu, mbar_wait(&bar[4], ph) && mbar_wait(&bar[9], ph));
  tc::fence_after();
  float *db2 = reinterpret_cast<float *>(smem + S::DB2P);
  if (ok) {
    // dA = Diag(beta) dL (strict lower) -> bf16 dA [r][j] and dA^T [j][r] operand tiles;
    // sum_j dL_rj A_rj -> dbeta
    float v[32];
    ld32(tl + T_DL + 32 * hf, v);
    tc::wait_ld();
    if (lane < 16) {
      const float br = sb[r64];
      float part = 0.f;
#pragma unroll
      for (int cb = 0; cb < 4; ++cb) {
        const int j0 = 32 * hf + 8 * cb;
        const float4 a0 = *reinterpret_cast<const float4 *>(smem + S::AS + tc::sw128_off32(64, r64, j0));
        const float4 a1 = *reinterpret_cast<const float4 *>(smem + S::AS + tc::sw128_off32(64, r64, j0 + 4));
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        float x8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float dl = j0 + e < r64 ? -v[8 * cb + e] : 0.f;
          part = fmaf(dl, av[e], part);
          x8[e] = br * dl;
        }
        *reinterpret_cast<uint4 *>(smem + S::DA + tc::sw128_off(64, r64, j0)) = tc::pack8(x8);
      }
      db2[hf * 64 + r64] = part;
    }
  }
  fence_proxy_async();
  tc::fence_before();
  if (!__syncthreads_and(ok)) return fail_out();
  tc::fence_after();
  {   // the next block's dO, T, S^T block 0 and Tb into the dO/A, T, X^T and dT tiles, free from here on
    if (tid == 32 && have_next) {
      const int nt0 = (int)nr.t0, narow = (int)nrid * 128;
      fence_proxy_async();
      mbar_expect_tx(&bar[10], 3 * 16384 + (TcRec::BYTES - TcRec::TB));
      bulk_g2s(smem + S::SS, (const char *)p.saved + nrid * 32768, 16384, &bar[10]);
      bulk_g2s(smem + S::TB, (const char *)p.img + nrid * TcRec::BYTES + TcRec::TB, TcRec::BYTES - TcRec::TB, &bar[10]);
      tc::tma_load_3d(smem + S::DO, &p.tm_do, 0, nh, nt0, &bar[10]);
      tc::tma_load_3d(smem + S::DO + 8192, &p.tm_do, 64, nh, nt0, &bar[10]);
      tc::tma_load_2d(smem + S::TK, &p.tm_aux, 0, narow + 64, &bar[10]);
      tc::tma_load_2d(smem + S::TK + 8192, &p.tm_aux, 32, narow + 64, &bar[10]);
    }
  }
  if (tid < ref.len) {   // ref.len <= 64
    const float *db1 = reinterpret_cast<const float *>(smem + S::DB1P);
    p.dbeta[(size_t)(ref.t0 + tid) * H + h] =
        ((db1[tid] + db1[64 + tid]) + (db1[128 + tid] + db1[192 + tid])) + (db2[tid] + db2[64 + tid]);
  }

  // ---------------------------------------------------------------- rounds (intra-chunk gradients)
  // Round t: P_tb = R_b^T dBm_tb^T, Q_tb = R_b^T dA_tb^T (b <= t), W_at = QL_a^T dBm_at + KL_a^T dA_at
  // (a >= t); M = 128 channels, N = K = 16. Rounds run t = 3, 2, 1, 0 (the dg suffix order) in two
  // TMEM buffers, the next but one issued as soon as a buffer is read out. Two threads issue each
  // round: part 0 the P products and the W sums of even a - t, part 1 the Q products and the rest.
  const uint32_t s_rf = smem_u32(smem + S::RF), s_qlf = smem_u32(smem + S::QLF), s_klf = smem_u32(smem + S::KLF),
                 s_dbm = smem_u32(smem + S::DBM), s_da = smem_u32(smem + S::DA);
  auto issue_round = [&](int t, uint32_t base, int part) {
    const uint32_t idn = tc::idesc_bf16_mn(128, 16, true, false), idw = tc::idesc_bf16_mn(128, 16, true, true);
    const uint32_t s_bb = part ? s_da : s_dbm, off = part ? 16 * (t + 1) : 0;
    for (int b = 0; b <= t; ++b)
      tc::mma_bf16(tmem + base + off + 16 * b, mnmaj(s_rf, b, 8192), tc::desc_sw128(s_bb + 2048 * t + 32 * b), idn, 0);
    for (int aa = t + part; aa < NSUB; aa += 2) {
      const uint32_t col = base + 32 * (t + 1) + 16 * (aa - t);
      // B(n = j in block t, k = r in block a) = dBm[r][j]: the rows r of the dBm (dA) tile, read MN-major
      tc::mma_bf16(tmem + col, mnmaj(s_qlf, aa, 8192), tc::desc_sw128_mn(s_dbm + 2048 * aa + 32 * t, 8192), idw, 0);
      tc::mma_bf16(tmem + col, mnmaj(s_klf, aa, 8192), tc::desc_sw128_mn(s_da + 2048 * aa + 32 * t, 8192), idw, 1);
    }
  };
  if (tid == 0 || tid == 32) {
    issue_round(3, T_R0, tid >> 5);
    tc::commit(&bar[5]);
    issue_round(2, T_R1, tid >> 5);
    tc::commit(&bar[6]);
  }
  RoundCtx rc{&p, &ref, smem, tl, row, hf, qw, lane, h, 0.f};
  {
    // sum_r dKh_rc Kh_rc (the e^{G_last} term of dg through Kh) over this thread's 32 rows, with Kh
    // in fp32 formed exactly as the round epilogues form R F_t: every row's dG takes this product
    // back out, so the two must agree to fp32 rounding (the record's bf16 Kh would leave an error
    // that does not shrink with dg)
    float v[32];
    ld32(tl + T_DKH + 32 * hf, v);
    tc::wait_ld();
    const bf16 *sk_ = (const bf16 *)(smem + S::KR);
    const float *csb = (const float *)(smem + (hf ? S::CSB : S::CSA)) + row;
    float cs = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int r = 32 * hf + i, t = r >> 4;
      const float kh = to_f(sk_[r * D + row]) * rk[r], yy = ex2(tot[t][row] - csb[i * 128]);
      cs += v[i] * fv[t][row] * (kh * yy);
    }
    reinterpret_cast<float *>(smem + S::CSUM)[hf * 128 + row] = cs;
  }
#pragma unroll 1
  for (int idx = 0; idx < NSUB; ++idx) {
    const uint32_t base = (idx & 1) ? T_R1 : T_R0;
    ok = mbar_wait(&bar[5 + idx], ph);
    tc::fence_before();
    if (!__syncthreads_and(ok)) return fail_out();
    tc::fence_after();
    if (idx == 0) {   // both halves of the Kh sum are in place after the barrier above
      const float *cs2 = reinterpret_cast<const float *>(smem + S::CSUM);
      rc.run = reinterpret_cast<const float *>(smem + S::TAIL)[row] + (cs2[row] + cs2[128 + row]);
    }
    round_epilogue(rc, NSUB - 1 - idx, base, [&]() {
      if ((tid == 0 || tid == 32) && idx < 2) {   // the round after next into this buffer
        issue_round(1 - idx, base, tid >> 5);
        tc::commit(&bar[7 + idx]);
      }
    });
  }
  tc::fence_before();
  __syncthreads();   // every tile of this block is consumed
  tc::fence_after();
  cur = nr;
  have_cur = have_next;
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, 512);
}

cudaError_t launch_bwd_chunk_tc(const BwdChunkParams &p, cudaStream_t s) {
  if (p.geo.max_chunks == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       BcSmem::BYTES);
  if (e != cudaSuccess) return e;
  const long long blocks = (long long)p.geo.max_chunks * p.geo.heads;   // head-fastest: see the kernel
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms < 1)
    sms = 1;
  const long long grid = blocks < sms ? blocks : sms;   // one persistent CTA per SM
  kda_bwd_chunk_tc_kernel<<<(unsigned)grid, BC_THREADS, BcSmem::BYTES, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
