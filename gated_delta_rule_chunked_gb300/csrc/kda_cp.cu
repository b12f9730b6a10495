// kda_cp.cu -- context parallelism: the segment-affine combine.
//
// A sequence split into P consecutive segments: each segment maps the state entering
// it affinely, S_out = M S_in + b (the KDA recurrence is linear in the state), with
// M its linear map on the key dimension and b its output from a zero state. Given
// every segment's (M, b), the state entering segment k follows by composing the maps
// in order: S_in[0] = h0, S_in[k+1] = M[k] S_in[k] + b[k]. One CTA per (sequence,
// head) runs that chain; the 128 x 128 fp32 state stays in shared memory and each
// thread accumulates an 8 x 8 tile of M S + b with fp32 FMAs (P products of
// 128^3, far from any bound next to the forward passes that produce M and b).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int CP_THREADS = 256;

__global__ void __launch_bounds__(CP_THREADS) kda_cp_combine_kernel(int P, int H, const float *M, const float *b,
                                                                     const float *h0, float *s_in) {
  extern __shared__ __align__(16) float cur[];   // [128][128]: the state entering the current segment
  const int sh = blockIdx.x, s = sh / H, h = sh % H;
  const int tid = threadIdx.x, i0 = 8 * (tid >> 4), j0 = 8 * (tid & 15);
  constexpr int SZ = D * D;
  for (int idx = tid; idx < SZ / 4; idx += CP_THREADS)
    reinterpret_cast<float4 *>(cur)[idx] =
        h0 ? reinterpret_cast<const float4 *>(h0 + (size_t)sh * SZ)[idx] : make_float4(0.f, 0.f, 0.f, 0.f);
  __syncthreads();
  for (int k = 0; k < P; ++k) {
    const size_t seg = ((size_t)s * P + k) * H + h;
    for (int idx = tid; idx < SZ / 4; idx += CP_THREADS)
      reinterpret_cast<float4 *>(s_in + seg * SZ)[idx] = reinterpret_cast<const float4 *>(cur)[idx];
    if (k + 1 == P) break;
    const float *Mk = M + seg * SZ, *bk = b + seg * SZ;
    float acc[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      const float4 x = *reinterpret_cast<const float4 *>(bk + (i0 + a) * D + j0);
      const float4 y = *reinterpret_cast<const float4 *>(bk + (i0 + a) * D + j0 + 4);
      acc[a][0] = x.x; acc[a][1] = x.y; acc[a][2] = x.z; acc[a][3] = x.w;
      acc[a][4] = y.x; acc[a][5] = y.y; acc[a][6] = y.z; acc[a][7] = y.w;
    }
#pragma unroll 1
    for (int m = 0; m < D; m += 4) {
      float mv[8][4];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        const float4 x = *reinterpret_cast<const float4 *>(Mk + (i0 + a) * D + m);
        mv[a][0] = x.x; mv[a][1] = x.y; mv[a][2] = x.z; mv[a][3] = x.w;
      }
#pragma unroll
      for (int mm = 0; mm < 4; ++mm) {
        const float4 x = *reinterpret_cast<const float4 *>(cur + (m + mm) * D + j0);
        const float4 y = *reinterpret_cast<const float4 *>(cur + (m + mm) * D + j0 + 4);
        const float sv[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
#pragma unroll
        for (int a = 0; a < 8; ++a)
#pragma unroll
          for (int c = 0; c < 8; ++c) acc[a][c] = fmaf(mv[a][mm], sv[c], acc[a][c]);
      }
    }
    __syncthreads();   // every thread is done reading the current state
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      *reinterpret_cast<float4 *>(cur + (i0 + a) * D + j0) = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
      *reinterpret_cast<float4 *>(cur + (i0 + a) * D + j0 + 4) = make_float4(acc[a][4], acc[a][5], acc[a][6], acc[a][7]);
    }
    __syncthreads();
  }
}

cudaError_t launch_cp_combine(int n_seqs, int n_segments, int heads, const float *M, const float *b, const float *h0,
                              float *s_in, cudaStream_t s) {
  const unsigned grid = (unsigned)((long long)n_seqs * heads);
  if (grid == 0) return cudaSuccess;
  constexpr int smem = D * D * (int)sizeof(float);
  const cudaError_t e = cudaFuncSetAttribute(kda_cp_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kda_cp_combine_kernel<<<grid, CP_THREADS, smem, s>>>(n_segments, heads, M, b, h0, s_in);
  return cudaGetLastError();
}

// Segment table: segment k of sequence i (k = 0..P-1) starts at s0 + 64 floor(nch k / P),
// capped at the sequence end s1 (nch = the sequence's chunk count); seg[N P] = the end.
__global__ void kda_cp_segments_kernel(const int *cu, int n_seqs, long long total, int P, int *seg) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long n = (long long)n_seqs * P;
  if (idx == 0) seg[n] = cu ? cu[n_seqs] : (int)total;
  if (idx >= n) return;
  const int i = (int)(idx / P), k = (int)(idx % P);
  const long long per = total / n_seqs;
  const long long s0 = cu ? cu[i] : per * i, s1 = cu ? cu[i + 1] : per * (i + 1);
  const long long nch = (s1 - s0 + CH - 1) / CH;
  const long long start = s0 + (long long)CH * ((nch * k) / P);
  seg[idx] = (int)(start < s1 ? start : s1);
}

cudaError_t launch_cp_segments(const int *cu, int n_seqs, long long total, int P, int *seg, cudaStream_t s) {
  const long long n = (long long)n_seqs * P;
  const unsigned blocks = (unsigned)((n + 255) / 256);
  kda_cp_segments_kernel<<<blocks ? blocks : 1, 256, 0, s>>>(cu, n_seqs, total, P, seg);
  return cudaGetLastError();
}

// Final state of each sequence = the final state of its last segment.
cudaError_t launch_cp_last(const float *hseg, int n_seqs, int P, int heads, float *hT, cudaStream_t s) {
  const size_t blk = (size_t)heads * D * D * sizeof(float);
  return cudaMemcpy2DAsync(hT, blk, hseg + (size_t)(P - 1) * heads * D * D, (size_t)P * blk, blk, (size_t)n_seqs,
                           cudaMemcpyDeviceToDevice, s);
}

}  // namespace kda
