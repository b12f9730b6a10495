// kda_scan_tc.cu -- the forward inter-chunk state passing on 5th-generation tensor cores.
//
// One CTA per (sequence, head): 4 state warps run the chain below, 4 io warps write
// the outputs. The 128x128 fp32 state lives in tensor
// memory for the whole sequence, transposed: TMEM lane m = value channel m,
// column n = key channel n (S^T). Thread t of warp w owns lane 32w + t, so every
// elementwise pass is a row pass. TMEM: two sets of 256 columns, [S^T | O^T | U^T]. Per 64-token chunk, with the record of the prep kernel
// (B1 = [Qt; -W], B2 = [Kh^T; Bm], Tb, gC; W = Tb Kt folds the intra-chunk
// WY/UT transform into one operand):
//
//   pass A : S^T -> bf16 operand tile (the saved chunk-start state is a bulk
//            copy of it); S^T <- S^T Diag(gC) in TMEM
//   phase 1: [O^T | U^T]  = S^T [Qt; -W]^T          (M=128, N=128, K=128)
//            U^T         += V^T Tb^T                 (M=128, N=64,  K=64; V^T read MN-major
//                                                     straight from the TMA boxes of V's rows)
//   pass B : U^T -> bf16 operand tile
//   phase 2: [S^T | O^T] += U^T [Kh^T; Bm]^T         (M=128, N=192, K=64)
// TMEM holds two sets of [S^T | O^T | U^T], alternating per chunk, so the previous
// chunk's O^T is written out while this chunk's phase 1 runs.
//
// i.e. U = Tb (V - Kt S), O = Qt S + Bm U, S <- gC*S + Kh^T U. A ninth warp issues
// phase 1: V^T Tb^T as soon as the values land (it does not need the state), the K-block
// of the state product that pass A has finished while pass A does the other, so only the
// last four MMAs wait for the whole of pass A; thread 0 issues phase 2. Completion is
// signalled through mbarriers (tcgen05.commit). The next
// chunk's record arrives by TMA bulk copy into the second of two buffers, and
// the next chunk's values arrive by TMA as soon as phase 1 has read this chunk's. Every wait
// is bounded; on a timeout the kernel reports KDA_ERR_TIMEOUT, frees its tensor
// memory and returns.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_tc05.cuh"

namespace kda {

struct TcScanSmem {
  static constexpr int RECS = (TcRec::BYTES + 1023) / 1024 * 1024;
  static constexpr int REC0 = 0, REC1 = RECS;
  static constexpr int AS = 2 * RECS;        // S^T bf16 [128][K=128]: two 16 KB blocks (also the saved state)
  static constexpr int AU = AS + 32768;      // U^T bf16 [128][K=64]; raw value rows before pass B
  static constexpr int AV = AU + 16384;      // V [64 tok][128] bf16 as two 64-channel SW128 boxes (V^T MN-major)
  static constexpr int OST = AV + 16384;     // staging [64 tok][128] bf16: raw values in, outputs out (io warps)
  static constexpr int BAR = OST + 16384;    // 6 mbarriers (see the kernel)
  static constexpr int TSLOT = BAR + 64;
  static constexpr int BYTES = TSLOT + 32 + 1024;   // + alignment slack
};

__device__ __forceinline__ void tc_issue_record(char *dst, const char *src, uint64_t *bar) {
  fence_proxy_async();
  mbar_expect_tx(bar, TcRec::BYTES);
  bulk_g2s(dst, src, TcRec::BYTES, bar);
}

// V rows of chunk j (two 64-channel boxes, 128-byte swizzle) into the V tile, completing on bar.
__device__ __forceinline__ void tc_issue_v(char *dst, const FwdScanParams &p, int h, long long t0, uint64_t *bar) {
  mbar_expect_tx(bar, 16384);
  tc::tma_load_3d(dst, &p.tm_v, 0, h, (int)t0, bar);
  tc::tma_load_3d(dst + 8192, &p.tm_v, 64, h, (int)t0, bar);
}

constexpr int FS_THREADS = 288;   // 4 state warps, 4 io warps, 1 phase-1 issuer warp

__global__ void __launch_bounds__(FS_THREADS, 1) kda_fwd_scan_tc_kernel(const __grid_constant__ FwdScanParams p) {
  using S = TcScanSmem;
  extern __shared__ __align__(1024) char smem_raw[];
  // operand tiles need 1024-byte alignment in the shared window
  char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  // paired launch: even CTAs run their unit from the identity with zero values (the state map of
  // the unit), odd CTAs run it as given
  const bool paired = p.hT_ident != nullptr, ident_cta = paired && (blockIdx.x & 1u) == 0;
  const unsigned unit = paired ? blockIdx.x >> 1 : blockIdx.x;
  const int H = p.geo.heads, h = (int)(unit % (unsigned)H), seq = (int)(unit / (unsigned)H);
  const long long s0 = p.geo.cu[seq], s1 = p.geo.cu[seq + 1];
  const int nch = (int)((s1 - s0 + CH - 1) / CH), cbase = p.geo.chunk_off[seq];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool io = warp >= 4 && warp < 8;      // warps 4..7: values in, outputs out; warp 8: phase-1 MMAs
  const int row = tid & 127, qw = warp & 3;   // row = TMEM lane = value channel
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::BAR);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + S::TSLOT);
  const bf16 *v = ident_cta ? nullptr : (const bf16 *)p.v;
  bf16 *o = ident_cta ? nullptr : (bf16 *)p.o;
  float *hT = ident_cta ? p.hT_ident : p.hT;
  const bool h0_identity = ident_cta || p.h0_identity;
  const float *h0 = ident_cta ? nullptr : p.h0;
  bf16 *saved = ident_cta ? nullptr : (bf16 *)p.saved;
  const size_t sh = (size_t)seq * H + h;

  // bar[0..1]: record buffers; bar[2]: phase 1 done; bar[3]: phase 2 done (MMA commits);
  // bar[4]: the V tile of a chunk landed (TMA); bar[5]: O^T of a chunk read out (128 io arrivals);
  // bar[6], bar[7]: pass A has written K-block 0, then all, of the S^T operand tile (128 state
  // arrivals each, the second also after a short last chunk's value rows are zeroed)
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
    mbar_init(&bar[5], 128);
    mbar_init(&bar[6], 128);
    mbar_init(&bar[7], 128);
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tl = tmem + ((uint32_t)(32 * qw) << 16);   // this warp's lane quarter
  // Two TMEM sets of [S^T | O^T | U^T] (128 + 64 + 64 columns) at 0 and 256; chunk j
  // works in set j & 1: pass A reads its start state from the other set and writes the
  // decayed state here, phase 2 accumulates [S^T | O^T] here in one N = 192 product, and
  // O^T of chunk j survives while chunk j + 1 runs in the other set.
  auto set_of = [](int j) -> uint32_t { return 256u * (uint32_t)(j & 1); };
  auto colO = [&](int j) -> uint32_t { return set_of(j) + 128u; };
  auto rec_of = [&](int j) { return (const char *)p.img + ((size_t)(cbase + j) * H + h) * TcRec::BYTES; };

  const uint64_t lim = p.wait_ns;   // limit of every bounded wait below
  bool ok = true;
  if (warp < 4) {
    // ------------------------------------------------------------ state warps
    // initial state S^T[dv][dk] = h0[dk][dv], in the set chunk 0 reads from
    {
      float buf[16];
#pragma unroll
      for (int cb = 0; cb < 8; ++cb) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          buf[i] = h0_identity ? (16 * cb + i == row ? 1.f : 0.f)
                               : (h0 ? h0[(sh * 128 + 16 * cb + i) * 128 + row] : 0.f);
        tc::st16(tl + set_of(1) + 16 * cb, buf);
      }
      tc::wait_st();
    }
    // shared-memory descriptors: the start-address field takes byte offsets >> 4 directly
    const uint64_t d_as = tc::desc_sw128(smem_u32(smem + S::AS)), d_au = tc::desc_sw128(smem_u32(smem + S::AU));
    const uint64_t d_rec0 = tc::desc_sw128(smem_u32(smem + S::REC0)), d_rec1 = tc::desc_sw128(smem_u32(smem + S::REC1));
    // Testing aid (p.starve): CTA 0 issues none of its first copies, so nothing of it is in
    // flight and its first waits run out after p.wait_ns; it reports KDA_ERR_TIMEOUT and leaves.
    if (tid == 0 && nch > 0 && !(p.starve && blockIdx.x == 0)) {
      tc_issue_record(smem + S::REC0, rec_of(0), &bar[0]);
      if (nch > 1) tc_issue_record(smem + S::REC1, rec_of(1), &bar[1]);
      if (v) tc_issue_v(smem + S::AV, p, h, s0, &bar[4]);
    }
    if (!v) {   // zero values: the V tile stays zero
      for (int idx = tid; idx < 16384 / 16; idx += 128)
        *reinterpret_cast<uint4 *>(smem + S::AV + 16 * idx) = make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async();
    }
    int done = 0;   // chunks whose phase 2 was issued
    for (int j = 0; j < nch; ++j) {
      const int b = j & 1;
      char *rb = smem + (b ? S::REC1 : S::REC0);
      ok &= mbar_wait(&bar[b], (j >> 1) & 1, lim);
      if (j > 0) ok &= mbar_wait(&bar[3], (j - 1) & 1, lim);
      if (tid == 32 && saved) bulk_wait_read();   // the previous saved-state copy has read the S^T tile
      tc::fence_after();
      if (!named_sync_and(1, 128, ok)) break;
      // the other record buffer's last reader (phase 2 of the previous chunk) has finished:
      // fetch the next chunk's record now, a whole chunk step ahead
      if (tid == 32 && j >= 1 && j + 1 < nch)
        tc_issue_record(smem + ((j + 1) & 1 ? S::REC1 : S::REC0), rec_of(j + 1), &bar[(j + 1) & 1]);
      // pass A: state -> operand tile, decayed state into this chunk's set
      {
        const float *gC = reinterpret_cast<const float *>(rb + TcRec::GC);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {   // 64 key channels at a time, one TMEM round trip each
          uint32_t r[64];
          tc::ld64(tl + set_of(j + 1) + 64 * hb, r);
          tc::wait_ld();
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) {
            float buf[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) buf[i] = __uint_as_float(r[16 * cb + i]);
            const int k0 = 64 * hb + 16 * cb;
            *reinterpret_cast<uint4 *>(smem + S::AS + tc::sw128_off(128, row, k0)) = tc::pack8(buf);
            *reinterpret_cast<uint4 *>(smem + S::AS + tc::sw128_off(128, row, k0 + 8)) = tc::pack8(buf + 8);
#pragma unroll
            for (int i = 0; i < 16; ++i) buf[i] *= gC[k0 + i];
            tc::st16(tl + set_of(j) + k0, buf);
          }
          if (hb == 0) {   // K-block 0 of the operand tile is written: the issuer may start on it
            fence_proxy_async();
            tc::fence_before();
            mbar_arrive(&bar[6]);
          }
        }
        tc::wait_st();
      }
      if (v) {   // chunk j's V tile (issued a chunk step ago); a sequence's last chunk: rows past its end zeroed
        ok &= mbar_wait(&bar[4], j & 1, lim);
        const int clen = (int)(s1 - (s0 + (long long)j * CH) < CH ? s1 - (s0 + (long long)j * CH) : CH);
        if (clen < CH && ok)
          for (int idx = tid; idx < (CH - clen) * 16; idx += 128) {
            const int r = clen + (idx >> 4), c = idx & 15;
            *reinterpret_cast<uint4 *>(smem + S::AV + (c >> 3) * 8192 + r * 128 + 16 * (c & 7)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
      }
      // the whole operand tile (and a short chunk's zeroed value rows) is in place: the issuer
      // finishes phase 1
      fence_proxy_async();
      tc::fence_before();
      mbar_arrive(&bar[7]);
      ok &= mbar_wait(&bar[2], j & 1, lim);
      tc::fence_after();
      if (tid == 32) {
        // the next chunk's values first, then the chunk-start state, which leaves as one bulk
        // copy of the operand tile (it has until the next pass A to read the tile)
        if (v && j + 1 < nch) tc_issue_v(smem + S::AV, p, h, s0 + (long long)(j + 1) * CH, &bar[4]);
        if (saved) {
          bulk_s2g(saved + ((size_t)(cbase + j) * H + h) * 128 * 128, smem + S::AS, 32768);
          bulk_commit();
        }
      }
      // pass B: U^T -> operand tile
      {
        uint32_t r[64];
        tc::ld64(tl + colO(j) + 64, r);
        tc::wait_ld();
#pragma unroll
        for (int cb = 0; cb < 8; ++cb) {
          float buf[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) buf[i] = __uint_as_float(r[8 * cb + i]);
          *reinterpret_cast<uint4 *>(smem + S::AU + tc::sw128_off(128, row, 8 * cb)) = tc::pack8(buf);
        }
      }
      fence_proxy_async();
      tc::fence_before();
      if (!named_sync_and(1, 128, ok)) break;
      if (tid == 0) {
        // O^T of the previous chunk has been read out by the io warps. This keeps the io
        // warps at most one phase behind on every barrier they wait on (a parity wait
        // cannot tell two completed phases apart), and frees that set's O^T before the
        // next chunk's phase 1 overwrites it.
        const bool freed = j == 0 || mbar_wait(&bar[5], (j - 1) & 1, lim);
        tc::fence_after();
        ok &= freed;
        if (freed) {
          // [S^T | O^T] += U^T [Kh^T; Bm]^T in this chunk's set
          const uint64_t d_b2 = (b ? d_rec1 : d_rec0) + (TcRec::B2 >> 4);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_bf16(tmem + set_of(j), d_au + 2 * ks, d_b2 + 2 * ks, tc::idesc_bf16(128, 192), 1);
          tc::commit(&bar[3]);
        }
      }
      done = j + 1;
    }
    if (ok && done > 0) ok = mbar_wait(&bar[3], (done - 1) & 1, lim);
    tc::fence_after();
    if (named_sync_and(1, 128, ok)) {
      if (hT) {   // hT[dk][dv] = S^T[dv][dk], in the set of the last chunk
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t r[64];
          tc::ld64(tl + set_of(done + 1) + 64 * hb, r);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 64; ++i) hT[(sh * 128 + 64 * hb + i) * 128 + row] = __uint_as_float(r[i]);
        }
      }
    } else {
      report(p.status, ERR_TIMEOUT);
    }
    if (tid == 32 && saved) bulk_wait_all();   // saved states complete before the CTA leaves
  } else if (io) {
    // ------------------------------------------------------------ io warps
    // O^T of chunk j (TMEM) -> o. Each warp transposes its 32 value channels through its
    // own columns of the staging tile, then writes 64-byte row pieces with 16-byte stores.
    auto store_o = [&](int j) {
      const long long t0 = s0 + (long long)j * CH;
      const int clen = (int)(s1 - t0 < CH ? s1 - t0 : CH);
      uint32_t r[64];
      tc::ld64(tl + colO(j), r);
      tc::wait_ld();
#pragma unroll
      for (int i = 0; i < 64; ++i)
        *reinterpret_cast<bf16 *>(smem + S::OST + i * 256 + row * 2) = __float2bfloat16_rn(__uint_as_float(r[i]));
      __syncwarp();
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int tok = 8 * k + (lane >> 2), ch = 4 * qw + (lane & 3);   // 16-byte chunk ch of row tok
        if (o && tok < clen)
          *reinterpret_cast<uint4 *>(o + ((size_t)(t0 + tok) * H + h) * 128 + ch * 8) =
              *reinterpret_cast<const uint4 *>(smem + S::OST + tok * 256 + ch * 16);
      }
      __syncwarp();
    };
    for (int j = 0; j < nch; ++j) {
      ok &= mbar_wait(&bar[3], j & 1, lim);     // phase 2 of chunk j has completed O^T
      tc::fence_after();
      if (!named_sync_and(2, 128, ok)) break;
      store_o(j);
      named_sync(2, 128);                  // every warp is done with the staging tile
      tc::fence_before();
      mbar_arrive(&bar[5]);
    }
  } else if (lane == 0) {
    // ------------------------------------------------------------ phase-1 issuer (warp 8)
    // [O^T | U^T] = S^T [Qt; -W]^T + (0 | V^T Tb^T) of chunk j into its set. V^T Tb^T needs only
    // the values and the record, so it goes first (full chunks; a sequence's short last chunk
    // waits until the state warps have zeroed the rows past its end, bar[7]); K-block 0 of the
    // state product follows once pass A has written it (bar[6]), K-block 1 at bar[7]. The first
    // k-step is split into its O^T and U^T halves so that O^T is overwritten and U^T adds to
    // the values' product. Every wait is bounded; a timeout ends the loop (the state warps'
    // own bounded wait on bar[2] then reports it).
    const uint64_t d_as = tc::desc_sw128(smem_u32(smem + S::AS));
    const uint64_t d_rec0 = tc::desc_sw128(smem_u32(smem + S::REC0)), d_rec1 = tc::desc_sw128(smem_u32(smem + S::REC1));
    const uint64_t idesc_v = tc::idesc_bf16_mn(128, 64, true, false);
    auto v_products = [&](uint32_t dO, uint64_t d_tb, bool first) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        tc::mma_bf16(dO + 64, tc::desc_sw128_mn(smem_u32(smem + S::AV) + 2048u * ks, 8192), d_tb + 2 * ks, idesc_v,
                     !(first && ks == 0));
    };
    for (int j = 0; j < nch; ++j) {
      const int b = j & 1;
      const long long t0 = s0 + (long long)j * CH;
      const bool early_v = v && s1 - t0 >= CH;
      const uint64_t d_rb = b ? d_rec1 : d_rec0, d_b1 = d_rb + (TcRec::B1 >> 4), d_tb = d_rb + (TcRec::TB >> 4);
      const uint32_t dO = tmem + colO(j);
      if (!mbar_wait(&bar[b], (j >> 1) & 1, lim)) break;
      if (early_v) {
        if (!mbar_wait(&bar[4], j & 1, lim)) break;
        tc::fence_after();
        v_products(dO, d_tb, true);
      }
      if (!mbar_wait(&bar[6], j & 1, lim)) break;
      tc::fence_after();
      tc::mma_bf16(dO, d_as, d_b1, tc::idesc_bf16(128, 64), 0);                              // O^T half
      tc::mma_bf16(dO + 64, d_as, d_b1 + (8192 >> 4), tc::idesc_bf16(128, 64), early_v ? 1u : 0u);   // U^T half
#pragma unroll
      for (int ks = 1; ks < 4; ++ks)
        tc::mma_bf16(dO, d_as + ((32 * ks) >> 4), d_b1 + ((32 * ks) >> 4), tc::idesc_bf16(128, 128), 1);
      if (!mbar_wait(&bar[7], j & 1, lim)) break;
      tc::fence_after();
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t off = (16384 + 32 * ks) >> 4;
        tc::mma_bf16(dO, d_as + off, d_b1 + off, tc::idesc_bf16(128, 128), 1);
      }
      if (v && !early_v) v_products(dO, d_tb, false);
      tc::commit(&bar[2]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, 512);
}

cudaError_t launch_fwd_scan_tc(const FwdScanParams &p, cudaStream_t s) {
  const long long units = (long long)p.geo.n_seqs * p.geo.heads;
  if (units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kda_fwd_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcScanSmem::BYTES);
  if (e != cudaSuccess) return e;
  const long long ctas = units * (p.hT_ident ? 2 : 1);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kda_fwd_scan_tc_kernel<<<(unsigned)ctas, FS_THREADS, TcScanSmem::BYTES, s>>>(p);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- backward
// Reverse dS scan, same arrangement (4 state warps, 4 io warps writing dv; dO arrives
// by TMA as two 64-channel boxes of 128-byte-swizzled rows, read MN-major as dO^T): dS^T in TMEM columns [0,128), dU^T in
// [128,192), dV^T in [192,256). Per chunk (last to first), with the forward's record
// read MN-major (its [Qt; -W], [Kh^T; Bm] and Tb tiles are the transposes of what the
// products here take K-major):
//   pass A : dS^T -> bf16 operand tile (saved as the chunk-end dS by one bulk copy);
//            dS^T <- dS^T Diag(gC)
//   phase 1: dU^T  = dO^T Bm + dS^T Kh^T           (M=128, N=64, K=64 + 128)
//   pass B : dU^T -> operand tile (K-block 1 of A2)
//   phase 2: dS^T += [dO^T | dU^T] [Qt^T | -W^T]^T  (M=128, N=128, K=128)
//            dV^T  = dU^T Tb                        (M=128, N=64,  K=64)
// i.e. dU = Bm^T dO + Kh dS, dS <- gC*dS + Qt^T dO - W^T dU, dv = Tb^T dU.
struct TcBwdSmem {
  static constexpr int RECS = (TcRec::BYTES + 1023) / 1024 * 1024;
  static constexpr int REC0 = 0, REC1 = RECS;
  static constexpr int AS = 2 * RECS;        // dS^T bf16 [128][K=128]
  static constexpr int A2 = AS + 32768;      // K-block 0: dO [64 tok][128] as two SW128 boxes (dO^T MN-major);
                                             // K-block 1: dU^T bf16 [128][K=64] (K-major)
  static constexpr int DST = A2 + 32768;     // staging: dv rows out (io warps)
  static constexpr int BAR = DST + 16384;
  static constexpr int TSLOT = BAR + 64;   // 6 mbarriers (see the kernel)
  static constexpr int BYTES = TSLOT + 32 + 1024;
};

// dO rows of chunk j into K-block 0 of A2 (two 64-channel boxes), completing on bar.
__device__ __forceinline__ void tc_issue_do(char *dst, const BwdScanParams &p, int h, long long t0, uint64_t *bar) {
  mbar_expect_tx(bar, 16384);
  tc::tma_load_3d(dst, &p.tm_do, 0, h, (int)t0, bar);
  tc::tma_load_3d(dst + 8192, &p.tm_do, 64, h, (int)t0, bar);
}

__global__ void __launch_bounds__(256, 1) kda_bwd_scan_tc_kernel(const __grid_constant__ BwdScanParams p) {
  using S = TcBwdSmem;
  extern __shared__ __align__(1024) char smem_raw[];
  char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int H = p.geo.heads, h = blockIdx.x % H, seq = blockIdx.x / H;
  const long long s0 = p.geo.cu[seq], s1 = p.geo.cu[seq + 1];
  const int nch = (int)((s1 - s0 + CH - 1) / CH), cbase = p.geo.chunk_off[seq];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool io = warp >= 4;                  // warps 4..7: dO in, dv out
  const int row = tid & 127, qw = warp & 3;   // row = TMEM lane = value channel
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem + S::BAR);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + S::TSLOT);
  const size_t sh = (size_t)seq * H + h;

  // bar[0..1]: record buffers; bar[2]: phase 1 done; bar[3]: phase 2 done (MMA commits);
  // bar[4]: the dO tile of a chunk landed (TMA); bar[5]: dV^T of a chunk read out (128 io
  // arrivals); bar[6]: phase 2's products that read the dO tile done (MMA commit)
  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bar[i], 1);
    mbar_init(&bar[5], 128);
    mbar_init(&bar[6], 1);
    fence_mbar_init();
  }
  if (warp == 0) tc::alloc(tslot, 256);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t tl = tmem + ((uint32_t)(32 * qw) << 16);
  auto rec_of = [&](int j) { return (const char *)p.img + ((size_t)(cbase + j) * H + h) * TcRec::BYTES; };

  bool ok = true;
  if (!io) {
    // ------------------------------------------------------------ state warps
    auto issue = [&](char *dst, const char *src, uint64_t *b) {
      fence_proxy_async();
      mbar_expect_tx(b, TcRec::BYTES);
      bulk_g2s(dst, src, TcRec::BYTES, b);
    };
    // initial dS^T[dv][dk] = dhT[dk][dv]
    {
      float buf[16];
#pragma unroll
      for (int cb = 0; cb < 8; ++cb) {
#pragma unroll
        for (int i = 0; i < 16; ++i) buf[i] = p.dhT ? p.dhT[(sh * 128 + 16 * cb + i) * 128 + row] : 0.f;
        tc::st16(tl + 16 * cb, buf);
      }
      tc::wait_st();
    }
    const uint64_t d_as = tc::desc_sw128(smem_u32(smem + S::AS)), d_a2 = tc::desc_sw128(smem_u32(smem + S::A2));
    if (tid == 0 && nch > 0) {
      tc_issue_do(smem + S::A2, p, h, s0 + (long long)(nch - 1) * CH, &bar[4]);
      issue(smem + S::REC0, rec_of(nch - 1), &bar[0]);
      if (nch > 1) issue(smem + S::REC1, rec_of(nch - 2), &bar[1]);
    }
    const uint32_t s_do = smem_u32(smem + S::A2);   // dO^T, MN-major: k-step ks at +2048 ks, channel atoms 8 KB apart
    int done = 0;
    for (int it = 0; it < nch; ++it) {
      const int j = nch - 1 - it, b = it & 1;
      char *rb = smem + (b ? S::REC1 : S::REC0);
      ok &= mbar_wait(&bar[b], (it >> 1) & 1);
      if (it > 0) ok &= mbar_wait(&bar[3], (it - 1) & 1);
      if (tid == 32) bulk_wait_read();   // the previous saved dS copy has read the dS^T tile
      tc::fence_after();
      if (!named_sync_and(1, 128, ok)) break;
      if (tid == 32 && it >= 1 && it + 1 < nch)   // next record, a whole chunk step ahead
        issue(smem + ((it + 1) & 1 ? S::REC1 : S::REC0), rec_of(j - 1), &bar[(it + 1) & 1]);
      if (tid == 64 && it + 2 < nch) {   // the chunk after that (record and dO) into L2
        prefetch_l2(rec_of(j - 2), TcRec::BYTES);
        tc::tma_prefetch_3d(&p.tm_do, 0, h, (int)(s0 + (long long)(j - 2) * CH));
        tc::tma_prefetch_3d(&p.tm_do, 64, h, (int)(s0 + (long long)(j - 2) * CH));
      }
      // pass A: dS^T -> operand tile, decayed dS^T back to TMEM
      {
        const float *gC = reinterpret_cast<const float *>(rb + TcRec::GC);
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t r[64];
          tc::ld64(tl + 64 * hb, r);
          tc::wait_ld();
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) {
            float buf[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) buf[i] = __uint_as_float(r[16 * cb + i]);
            const int k0 = 64 * hb + 16 * cb;
            *reinterpret_cast<uint4 *>(smem + S::AS + tc::sw128_off(128, row, k0)) = tc::pack8(buf);
            *reinterpret_cast<uint4 *>(smem + S::AS + tc::sw128_off(128, row, k0 + 8)) = tc::pack8(buf + 8);
#pragma unroll
            for (int i = 0; i < 16; ++i) buf[i] *= gC[k0 + i];
            tc::st16(tl + k0, buf);
          }
        }
        tc::wait_st();
      }
      {   // this chunk's dO tile; a sequence's last chunk (the first one here): rows past its end zeroed
        ok &= mbar_wait(&bar[4], it & 1);
        const long long t0 = s0 + (long long)j * CH;
        const int clen = (int)(s1 - t0 < CH ? s1 - t0 : CH);
        if (clen < CH && ok)
          for (int idx = tid; idx < (CH - clen) * 16; idx += 128) {
            const int r = clen + (idx >> 4), c = idx & 15;
            *reinterpret_cast<uint4 *>(smem + S::A2 + (c >> 3) * 8192 + r * 128 + 16 * (c & 7)) =
                make_uint4(0u, 0u, 0u, 0u);
          }
      }
      fence_proxy_async();
      tc::fence_before();
      if (!named_sync_and(1, 128, ok)) break;
      if (tid == 0) {
        tc::fence_after();
        {
          // B(n = j, k = r) = Bm[r][j]: rows r of the record's Bm tile -> MN-major
          const uint32_t s_b2 = smem_u32(rb) + TcRec::B2;
          constexpr uint32_t idn = tc::idesc_bf16_mn(128, 64, false, true);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_bf16(tmem + 128, tc::desc_sw128_mn(s_do + 2048 * ks, 8192),
                         tc::desc_sw128_mn(s_b2 + 16384 + 2048 * ks, 8192), tc::idesc_bf16_mn(128, 64, true, true), ks > 0);
          // B(n = j, k = dk) = Kh[j][dk] = Kh^T rows dk -> MN-major
#pragma unroll
          for (int kb = 0; kb < 2; ++kb)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              tc::mma_bf16(tmem + 128, d_as + ((kb * 16384 + 32 * ks) >> 4),
                           tc::desc_sw128_mn(s_b2 + 8192 * kb + 2048 * ks, 8192), idn, 1);
          tc::commit(&bar[2]);
        }
      } else if (tid == 32) {
        // the chunk-end dS leaves as one bulk copy of the operand tile
        bulk_s2g((bf16 *)p.dsaved + ((size_t)(cbase + j) * H + h) * 128 * 128, smem + S::AS, 32768);
        bulk_commit();
      }
      ok &= mbar_wait(&bar[2], it & 1);
      tc::fence_after();
      // pass B: dU^T -> K-block 1 of A2
      {
        uint32_t r[64];
        tc::ld64(tl + 128, r);
        tc::wait_ld();
#pragma unroll
        for (int cb = 0; cb < 8; ++cb) {
          float buf[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) buf[i] = __uint_as_float(r[8 * cb + i]);
          *reinterpret_cast<uint4 *>(smem + S::A2 + tc::sw128_off(128, row, 64 + 8 * cb)) = tc::pack8(buf);
        }
      }
      fence_proxy_async();
      tc::fence_before();
      if (!named_sync_and(1, 128, ok)) break;
      if (tid == 0) {
        // dV^T of the previous chunk has been read out by the io warps (frees its columns and
        // keeps the io warps at most one phase behind on every barrier they wait on)
        const bool freed = it == 0 || mbar_wait(&bar[5], (it - 1) & 1);
        tc::fence_after();
        ok &= freed;
        if (freed) {
          // B(n = dk, k = tok) = [Qt; -W][tok][dk]: rows tok of the record's B1 tile -> MN-major,
          // two 64-channel atoms 16 KB apart
          const uint32_t s_rb = smem_u32(rb);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)   // K-block 0: dO^T, MN-major
            tc::mma_bf16(tmem, tc::desc_sw128_mn(s_do + 2048 * ks, 8192),
                         tc::desc_sw128_mn(s_rb + TcRec::B1 + 2048 * ks, 16384), tc::idesc_bf16_mn(128, 128, true, true), 1);
          tc::commit(&bar[6]);             // the dO tile is read: the io warps refill it
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)   // K-block 1: dU^T, K-major
            tc::mma_bf16(tmem, d_a2 + ((16384 + 32 * ks) >> 4),
                         tc::desc_sw128_mn(s_rb + TcRec::B1 + 8192 + 2048 * ks, 16384),
                         tc::idesc_bf16_mn(128, 128, false, true), 1);
          // B(n = j, k = r) = Tb[r][j]: rows r of the record's Tb tile -> MN-major
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            tc::mma_bf16(tmem + 192, d_a2 + (16384 >> 4) + 2 * ks, tc::desc_sw128_mn(s_rb + TcRec::TB + 2048 * ks, 8192),
                         tc::idesc_bf16_mn(128, 64, false, true), ks > 0);
          tc::commit(&bar[3]);
        }
      }
      done = it + 1;
    }
    if (ok && done > 0) ok = mbar_wait(&bar[3], (done - 1) & 1);
    tc::fence_after();
    if (named_sync_and(1, 128, ok)) {
      if (p.dh0) {   // dh0[dk][dv] = dS^T[dv][dk]
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t r[64];
          tc::ld64(tl + 64 * hb, r);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 64; ++i) p.dh0[(sh * 128 + 64 * hb + i) * 128 + row] = __uint_as_float(r[i]);
        }
      }
    } else {
      report(p.status, ERR_TIMEOUT);
    }
    if (tid == 32) bulk_wait_all();   // saved dS complete before the CTA leaves
  } else {
    // ------------------------------------------------------------ io warps
    // dV^T (TMEM) -> dv rows of chunk j (fp32). Each warp transposes its 32 value channels
    // through its own 4 KB of the staging tile, 32 tokens at a time, and writes 128-byte
    // row pieces with 16-byte stores.
    auto store_dv = [&](int j) {
      const long long t0 = s0 + (long long)j * CH;
      const int clen = (int)(s1 - t0 < CH ? s1 - t0 : CH);
      uint32_t r[64];
      tc::ld64(tl + 192, r);
      tc::wait_ld();
      float *wst = reinterpret_cast<float *>(smem + S::DST + qw * 4096);   // [32 tok][32 channels]
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int i = 0; i < 32; ++i) wst[i * 32 + lane] = __uint_as_float(r[32 * half + i]);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int tok = 4 * k + (lane >> 3), ch = lane & 7, gt = 32 * half + tok;
          if (gt < clen)
            *reinterpret_cast<float4 *>(p.dv + ((size_t)(t0 + gt) * H + h) * 128 + 32 * qw + 4 * ch) =
                *reinterpret_cast<const float4 *>(wst + tok * 32 + 4 * ch);
        }
        __syncwarp();
      }
    };
    for (int it = 0; it < nch; ++it) {
      const int j = nch - 1 - it;
      if (it + 1 < nch) {   // phase 2 has read this chunk's dO tile: the next chunk's dO into it
        const bool rd = mbar_wait(&bar[6], it & 1);
        ok &= rd;
        if (tid == 128 && rd) {
          tc::fence_after();
          tc_issue_do(smem + S::A2, p, h, s0 + (long long)(j - 1) * CH, &bar[4]);
        }
      }
      ok &= mbar_wait(&bar[3], it & 1);   // phase 2 of this chunk: dV^T is final
      tc::fence_after();
      if (!named_sync_and(2, 128, ok)) break;
      store_dv(j);
      named_sync(2, 128);                  // every warp is done with the staging tile
      tc::fence_before();
      mbar_arrive(&bar[5]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 0) tc::dealloc(tmem, 256);
}

cudaError_t launch_bwd_scan_tc(const BwdScanParams &p, cudaStream_t s) {
  const long long units = (long long)p.geo.n_seqs * p.geo.heads;
  if (units == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kda_bwd_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcBwdSmem::BYTES);
  if (e != cudaSuccess) return e;
  kda_bwd_scan_tc_kernel<<<(unsigned)units, 256, TcBwdSmem::BYTES, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
