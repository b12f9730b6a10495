// kda_common.cuh -- shared device helpers of the KDA kernels (sm_103a).
//
// * swizzled shared-memory tiles (16-byte chunks XOR-permuted by row so that
//   8-row ldmatrix accesses hit distinct banks),
// * warp-level tile GEMMs with one accumulator layout for two element types:
//   bf16 tiles use ldmatrix + mma.sync m16n8k16 (fp32 accumulate); fp32 tiles
//   use an FMA loop that fills the same m16n8 fragment positions, which gives
//   the fp32-I/O path full fp32 products,
// * mbarrier + cp.async.bulk (TMA bulk copy) helpers with bounded waits.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {

constexpr int D = 128;       // dk = dv
constexpr int CH = 64;       // chunk length
constexpr int SUB = 16;      // sub-block of the gated Gram factorisation
constexpr int NSUB = CH / SUB;
constexpr float LOG2E = 1.4426950408889634f;
constexpr int ERR_TIMEOUT = 4;   // matches KDA_ERR_TIMEOUT
constexpr int KDA_ERR_INVALID_ARG_CODE = 1;   // matches KDA_ERR_INVALID_ARG

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- tiles
// Physical 16-byte chunk of logical chunk `ch` in row `row` for rows of CPR chunks.
template <int CPR>
__device__ __forceinline__ int swz(int row, int ch) {
  if constexpr (CPR >= 8) return (ch & ~7) | ((ch ^ row) & 7);
  else if constexpr (CPR == 4) return ch ^ ((row >> 1) & 3);
  else if constexpr (CPR == 2) return ch ^ ((row >> 2) & 1);
  else return ch;
}

// A row-major tile of element type E whose rows hold LD elements, swizzled.
template <typename E, int LD>
struct Tile {
  static constexpr int EPC = 16 / (int)sizeof(E);   // elements per 16-byte chunk
  static constexpr int CPR = LD / EPC;              // chunks per row
  static constexpr int BYTES_PER_ROW = LD * (int)sizeof(E);
  E *p;
  __device__ __forceinline__ Tile(E *ptr) : p(ptr) {}
  __device__ __forceinline__ int off(int r, int c) const {
    return r * LD + swz<CPR>(r, c / EPC) * EPC + (c % EPC);
  }
  __device__ __forceinline__ E *at(int r, int c) const { return p + off(r, c); }
};

// A bf16 tile of R rows x 128 columns in the tcgen05 K-major 128-byte-swizzle
// layout: two 64-column blocks of R rows x 128 bytes; inside a row, 16-byte chunk
// c sits at c ^ (row % 8). This is the layout of the scans' operand tiles and of
// the chunk states they save, so a saved state is one contiguous bulk copy.
template <int R>
struct TileSW {
  bf16 *p;
  __device__ __forceinline__ TileSW(bf16 *ptr) : p(ptr) {}
  __device__ __forceinline__ int off(int r, int c) const {
    return (c >> 6) * R * 64 + r * 64 + ((((c & 63) >> 3) ^ (r & 7)) << 3) + (c & 7);
  }
  __device__ __forceinline__ bf16 *at(int r, int c) const { return p + off(r, c); }
};

__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }
template <typename E> __device__ __forceinline__ E from_f(float x);
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }

// Store two adjacent elements (c even) of a tile.
__device__ __forceinline__ void st2(bf16 *p, float a, float b) {
  *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(a, b);
}
__device__ __forceinline__ void st2(float *p, float a, float b) {
  *reinterpret_cast<float2 *>(p) = make_float2(a, b);
}
__device__ __forceinline__ float2 ld2(const bf16 *p) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(p));
}
__device__ __forceinline__ float2 ld2(const float *p) { return *reinterpret_cast<const float2 *>(p); }

// ---------------------------------------------------------------- mma.sync
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t &r0, uint32_t &r1, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t &r0, uint32_t &r1, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];\n"
               : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// TF32 tensor-core product m16n8k8 (fp32 accumulate). Fragments (g = lane/4, q = lane%4):
//   a0 = A[g][q], a1 = A[g+8][q], a2 = A[g][q+4], a3 = A[g+8][q+4];  b0 = B[q][g], b1 = B[q+4][g].
__device__ __forceinline__ uint32_t tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ void mma1688(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Accumulator fragment of an m16n8 tile for lane (g = lane/4, q = lane%4):
//   c[0] = (g, 2q), c[1] = (g, 2q+1), c[2] = (g+8, 2q), c[3] = (g+8, 2q+1).
//
// wgemm: acc[nt] += A[m0:m0+16, k0:k1] * B[k0:k1, n0+8nt : n0+8nt+8] for nt < NT.
//   AK: A stored [m][k] (true) or [k][m] (false);
//   BK: B stored [n][k] (true) or [k][n] (false).
// k0, k1 are multiples of 16. A and B are bf16 tiles (Tile<bf16, LD> or TileSW<R>:
// any tile whose 8 consecutive columns from a multiple of 8 are 16 contiguous bytes).
template <bool AK, bool BK, int NT, class TA, class TB>
__device__ __forceinline__ void wgemm(float (&acc)[NT][4], TA A, int m0, TB B, int n0, int k0, int k1) {
  const int lane = threadIdx.x & 31;
  const int i = lane >> 3, r8 = lane & 7;
#pragma unroll 2
  for (int kk = k0; kk < k1; kk += 16) {
    uint32_t a[4];
    if constexpr (AK) {
      ldsm_x4(a, smem_u32(A.at(m0 + r8 + (i & 1) * 8, kk + (i >> 1) * 8)));
    } else {
      ldsm_x4_t(a, smem_u32(A.at(kk + (i >> 1) * 8 + r8, m0 + (i & 1) * 8)));
    }
#pragma unroll
    for (int nt = 0; nt + 1 < NT; nt += 2) {
      uint32_t b[4];
      if constexpr (BK) {
        ldsm_x4(b, smem_u32(B.at(n0 + nt * 8 + (i >> 1) * 8 + r8, kk + (i & 1) * 8)));
      } else {
        ldsm_x4_t(b, smem_u32(B.at(kk + (i & 1) * 8 + r8, n0 + nt * 8 + (i >> 1) * 8)));
      }
      mma16816(acc[nt], a, b[0], b[1]);
      mma16816(acc[nt + 1], a, b[2], b[3]);
    }
    if constexpr (NT & 1) {
      constexpr int nt = NT - 1;
      uint32_t b0, b1;
      const int j = i & 1;
      if constexpr (BK) {
        ldsm_x2(b0, b1, smem_u32(B.at(n0 + nt * 8 + r8, kk + j * 8)));
      } else {
        ldsm_x2_t(b0, b1, smem_u32(B.at(kk + j * 8 + r8, n0 + nt * 8)));
      }
      mma16816(acc[nt], a, b0, b1);
    }
  }
}

// fp32 tiles: same fragment positions, exact fp32 FMAs, in k order. With B stored [k][n] a
// lane's two columns 2q, 2q+1 sit in one 16-byte chunk of the row, so they come in one 8-byte
// load; with A stored [m][k] the values at k and k + 1 (k even) do too, so A is read two k at a
// time (k0 and k1 even).
template <bool AK, bool BK, int NT, int LDA, int LDB>
__device__ __forceinline__ void wgemm(float (&acc)[NT][4], Tile<float, LDA> A, int m0, Tile<float, LDB> B,
                                      int n0, int k0, int k1) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  auto step = [&](int k, float a0, float a1) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int n = n0 + nt * 8 + 2 * q;
      float b0, b1;
      if constexpr (BK) {
        b0 = *B.at(n, k);
        b1 = *B.at(n + 1, k);
      } else {
        const float2 bb = *reinterpret_cast<const float2 *>(B.at(k, n));
        b0 = bb.x;
        b1 = bb.y;
      }
      acc[nt][0] = fmaf(a0, b0, acc[nt][0]);
      acc[nt][1] = fmaf(a0, b1, acc[nt][1]);
      acc[nt][2] = fmaf(a1, b0, acc[nt][2]);
      acc[nt][3] = fmaf(a1, b1, acc[nt][3]);
    }
  };
  if constexpr (AK) {
    for (int k = k0; k < k1; k += 2) {
      const float2 x0 = *reinterpret_cast<const float2 *>(A.at(m0 + g, k));
      const float2 x1 = *reinterpret_cast<const float2 *>(A.at(m0 + g + 8, k));
      step(k, x0.x, x1.x);
      step(k + 1, x0.y, x1.y);
    }
  } else {
    for (int k = k0; k < k1; ++k) step(k, *A.at(k, m0 + g), *A.at(k, m0 + g + 8));
  }
}

// Two fp32 products with one B operand in one k loop (each accumulator in k order, as two
// wgemm calls): acc1 += A1 B, acc2 += A2 B, A1 and A2 stored [m][k], B stored [k][n]; the B
// values are loaded once for both. k0 and k1 even.
template <int NT, int LDA, int LDB>
__device__ __forceinline__ void wgemm2(float (&acc1)[NT][4], float (&acc2)[NT][4], Tile<float, LDA> A1,
                                       Tile<float, LDA> A2, int m0, Tile<float, LDB> B, int n0, int k0, int k1) {
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  for (int k = k0; k < k1; k += 2) {
    const float2 x0 = *reinterpret_cast<const float2 *>(A1.at(m0 + g, k));
    const float2 x1 = *reinterpret_cast<const float2 *>(A1.at(m0 + g + 8, k));
    const float2 y0 = *reinterpret_cast<const float2 *>(A2.at(m0 + g, k));
    const float2 y1 = *reinterpret_cast<const float2 *>(A2.at(m0 + g + 8, k));
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const float a0 = kk ? x0.y : x0.x, a1 = kk ? x1.y : x1.x, c0 = kk ? y0.y : y0.x, c1 = kk ? y1.y : y1.x;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float2 bb = *reinterpret_cast<const float2 *>(B.at(k + kk, n0 + nt * 8 + 2 * q));
        acc1[nt][0] = fmaf(a0, bb.x, acc1[nt][0]);
        acc1[nt][1] = fmaf(a0, bb.y, acc1[nt][1]);
        acc1[nt][2] = fmaf(a1, bb.x, acc1[nt][2]);
        acc1[nt][3] = fmaf(a1, bb.y, acc1[nt][3]);
        acc2[nt][0] = fmaf(c0, bb.x, acc2[nt][0]);
        acc2[nt][1] = fmaf(c0, bb.y, acc2[nt][1]);
        acc2[nt][2] = fmaf(c1, bb.x, acc2[nt][2]);
        acc2[nt][3] = fmaf(c1, bb.y, acc2[nt][3]);
      }
    }
  }
}

template <int NT>
__device__ __forceinline__ void zero(float (&acc)[NT][4]) {
#pragma unroll
  for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
}

// ---------------------------------------------------------------- cp.async (LDGSTS)
// 16-byte global -> shared copy through the load/store units; `valid` bytes are
// read (0 or 16), the rest of the 16 is zero-filled. Completes at cp_async_wait_all.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int valid = 16) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(valid)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// ---------------------------------------------------------------- TMA bulk copies
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Global -> shared bulk copy; bytes and both addresses multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
// Shared -> global bulk copy (one thread); bytes and both addresses multiples of 16.
// Tracked per thread by bulk groups: bulk_commit() closes a group, bulk_wait_read()
// returns once every committed group has finished reading shared memory.
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
// Ask for `bytes` (a multiple of 16, from a 16-byte aligned address) of global memory to be
// brought into L2; nothing waits for it and no register or shared memory is held.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(__cvta_generic_to_global(src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Wait for phase `parity` of `bar`, giving up after ~2 s. Returns false on timeout.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;   // default limit of every bounded wait (about 2 s)

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns = WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Named barrier over `count` threads (a multiple of 32) of this CTA.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also returns the AND of `pred` over the participating threads.
__device__ __forceinline__ bool named_sync_and(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void report(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- chunk table
// Chunk c of the packed problem: sequence index, first token, valid length.
struct ChunkRef {
  int seq;
  long long t0;
  int len;
};

// chunk_off[i] = first global chunk of sequence i (prefix sum of ceil(L_i/64)),
// chunk_off[N] = number of chunks. Binary search for the owner of chunk c.
__device__ __forceinline__ bool chunk_lookup(const int *chunk_off, const int *cu, int n_seqs, int c,
                                             ChunkRef &ref) {
  if (c >= chunk_off[n_seqs]) return false;
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (chunk_off[mid] <= c) lo = mid; else hi = mid - 1;
  }
  const long long s0 = cu[lo], s1 = cu[lo + 1];
  ref.seq = lo;
  ref.t0 = s0 + (long long)(c - chunk_off[lo]) * CH;
  const long long rem = s1 - ref.t0;
  ref.len = rem < CH ? (int)rem : CH;
  return true;
}

}  // namespace kda
