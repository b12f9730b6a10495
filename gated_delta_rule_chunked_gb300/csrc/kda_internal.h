// kda_internal.h -- host-side launch interfaces between kda_api.cu and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

// Per-(chunk, head) record written by the chunk-prep kernel and read by the scans.
// Tiles are stored exactly as they sit in shared memory (swizzled), so a single
// bulk copy moves each of them. Element type E = bf16 (2 bytes) or float (4).
//   [Qt | Kt]  64x128  q^*exp(G), k^*exp(G)           region 1
//   [Tb]       64x64   T Diag(beta)                    region 2
//   [Bm]       64x64   masked gated q.k^T              region 3
//   [Kh | gC]  64x128  k^*exp(G_last-G); 128 fp32 exp(G_last)   region 4
struct ImgLayout {
  int esz;
  size_t qt, kt, tb, bm, kh, gc, bytes;
  __host__ __device__ explicit ImgLayout(int elem_size) : esz(elem_size) {
    const size_t t128 = (size_t)64 * 128 * elem_size, t64 = (size_t)64 * 64 * elem_size;
    qt = 0;
    kt = qt + t128;
    tb = kt + t128;
    bm = tb + t64;
    kh = bm + t64;
    gc = kh + t128;
    bytes = gc + 128 * sizeof(float);
  }
};

// Per-(chunk, head) record for the tcgen05 forward scan (bf16). Every tile is a
// K-major, 128-byte-swizzled operand image, so one bulk copy lands it ready for
// the tensor cores:
//   B1 [128 rows][K = 128 dk]: rows 0..63 Qt[tok], rows 64..127 -W[tok],  W = Tb Kt
//   B2 [192 rows][K = 64 tok]: rows 0..127 Kh^T[dk], rows 128..191 Bm[r]
//   TB [64 rows][K = 64]     : Tb[r][j]
//   GC 128 fp32              : exp(G_last)
struct TcRec {
  static constexpr int B1 = 0, B2 = 32768, TB = B2 + 24576, GC = TB + 8192, BYTES = GC + 512;
};

// Per-(chunk, head) Kt tile for the backward (bf16, training forward only): Kt[tok][dk]
// in the same K-major 128-byte-swizzle layout (two 8 KB blocks). Everything else the
// backward reads per chunk is in the forward record (TcRec), read MN-major where a
// product needs the other orientation.
struct KtRec {
  static constexpr int BYTES = 64 * 128 * 2;
};

struct SeqGeom {
  int n_seqs;
  long long total;
  int heads;
  int max_chunks;          // upper bound of the number of chunks (grid size)
  const int *cu;           // [N+1] device
  const int *chunk_off;    // [N+1] device, built by launch_chunk_table
};

struct PrepParams {
  // TMA maps of q, k (io type) and g (fp32): box 128 channels x 1 head x 64 tokens, plain rows
  CUtensorMap tm_q, tm_k, tm_g;
  SeqGeom geo;
  const void *q, *k;
  const float *g, *beta;
  float scale;
  void *img;               // [max_chunks][H] forward records: TcRec (bf16) or the tile record (fp32)
  float *aux;              // [max_chunks][H] x {A (strict lower), T} fp32 64x64 each, or NULL
  int tc_layout;           // bf16: bit 0 = write the tcgen05 forward record to img;
                           //       bit 1 = write the backward extras: Kt (img2) and aux
  void *img2;              // [max_chunks][H] KtRec tiles (bit 1)
  int *status;
  int prefetch_dist;       // tcgen05 prep: CTA b brings the staging boxes of CTA b + prefetch_dist into L2
};

struct FwdScanParams {
  SeqGeom geo;
  const void *v;
  const void *img;
  const float *h0;
  void *o;
  float *hT;
  void *saved;             // [max_chunks][H] chunk-start states S^T[v][k] as 128x128 E tiles
                           // (swizzled), or null
  int *status;
  int h0_identity;         // start every sequence from the identity state (h0 ignored)
  CUtensorMap tm_v;        // bf16 scan: v as boxes of 64 channels x 1 head x 64 tokens, 128-byte swizzle
  unsigned long long wait_ns;   // limit of every bounded wait of the tcgen05 scan
  int starve;              // testing aid: CTA 0 issues none of its first copies (its waits run out)
  float *hT_ident;         // tcgen05 scan, paired launch (non-null): CTA 2u runs unit u from the identity
                           // with zero values and no outputs (final states here), CTA 2u + 1 runs it as
                           // given; the two read the same records at about the same time (L2)
};

struct BwdScanParams {
  SeqGeom geo;
  const void *dO;
  const void *img;         // TcRec records (the forward's)
  const float *dhT;
  float *dv;
  float *dh0;
  void *dsaved;            // [max_chunks][H] 128x128 E tiles (swizzled): dS^T[v][k] at each chunk end
  int *status;
  CUtensorMap tm_do;       // dO as boxes of 64 channels x 1 head x 64 tokens, 128-byte swizzle
};

struct BwdChunkParams {
  // TMA maps: q, k, v (box 128 x 1 head x 64 tokens, plain rows), dO (box 64 x 1 x 64, 128-byte
  // swizzle), and the prep's A/T array as [items * 128 rows][64] fp32 (box 32 x 64, 128-byte swizzle)
  CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_aux;
  SeqGeom geo;
  const void *q, *k, *v, *dO;   // io type (bf16)
  const float *g, *beta;
  float scale;
  const void *img;              // [max_chunks][H] TcRec records (the forward's)
  const void *kt;               // [max_chunks][H] KtRec tiles
  const void *saved, *dsaved;   // [max_chunks][H] chunk-start states S^T, chunk-end dS^T (bf16 tiles)
  const float *aux;             // [max_chunks][H] x {A (strict lower), T} written by the prep kernel
  float *dq, *dk, *dg, *dbeta;
  int *status;
};

// fp32-I/O backward (kda_bwd_f32.cu). The records and {A, T} come from a prep run into the
// backward's workspace; `saved` holds the forward's chunk-start states S[k][v] and `dsaved`
// the dS scan's chunk-end gradients dS[k][v] (fp32 tiles, swizzled as Tile<float, 128>).
// The state-side kernel leaves dQt, dKt and dKh in the dq, dk and dg arrays and dBm, dA and
// dgC e^{G_last} in `scratch` (BWD_F32_SCRATCH floats per chunk-head); the intra-chunk
// kernel turns them into the final dq, dk and dg.
constexpr int BWD_F32_SCRATCH = 2 * 64 * 64 + 128;
struct BwdF32Params {
  SeqGeom geo;
  const float *q, *k, *v, *dO, *g, *beta;
  float scale;
  const void *img;              // [max_chunks][H] fp32 tile records (ImgLayout)
  const float *aux;             // [max_chunks][H] x {A, T}
  const float *saved, *dsaved;  // [max_chunks][H] 128 x 128
  float *dq, *dk, *dg, *dbeta;
  float *scratch;               // [max_chunks][H][BWD_F32_SCRATCH]
  int *status;
};

struct StepParams {
  int n_seqs, steps, heads;
  float scale;
  const void *q, *k, *v;
  const float *beta, *g;
  float *state;
  const int *accept_len;
  void *o;
  const int *state_indices;   // [N] pool slot per sequence, or null (slot = sequence)
  int n_slots;                // pool size with state_indices
  const int *first_slot;      // [N] leading padding slots, or null (0)
  int *status;
  int prefetch_dist;          // set by the launcher: CTA b prefetches the state of CTA b + prefetch_dist
};

struct AttnresParams {
  int S;
  long long T;
  int dim;
  float eps;
  const void *src[9];
  const float *w;
  void *out;
  float *alpha, *rstd, *logit;   // [T][S]
  int *status;                   // optional status word (a bounded wait that gave up)
  int nbuf;                      // backward: staging buffers per CTA (set by the launcher)
  const void *dout;
  void *dsrc[9];
  float *dw;
  float *partial;                // [backward CTAs][dim]
  long long prefetch_dist;       // forward: CTA b brings the source slices of CTA b + prefetch_dist into L2
};

cudaError_t launch_attnres_fwd(const AttnresParams &p, bool f32, cudaStream_t s);
cudaError_t launch_attnres_bwd(const AttnresParams &p, bool f32, cudaStream_t s);
int attnres_bwd_ctas(long long T, bool f32, int dim, int S);

cudaError_t launch_chunk_table(const int *cu_in, int n_seqs, long long total, int *cu_out,
                               int *chunk_off, cudaStream_t s);
cudaError_t launch_prep(const PrepParams &p, bool f32, cudaStream_t s);      // fp32 I/O (exact fp32 products)
cudaError_t launch_prep_tc(const PrepParams &p, cudaStream_t s);            // bf16 I/O (tcgen05)
cudaError_t launch_fwd_scan(const FwdScanParams &p, bool f32, int dv_slice, cudaStream_t s);
cudaError_t launch_fwd_scan_tc(const FwdScanParams &p, cudaStream_t s);
cudaError_t launch_bwd_scan_tc(const BwdScanParams &p, cudaStream_t s);
// Short convolution (kda_conv.cu). Forward: x, w, bias, st_in -> y, st_out. Backward adds
// dy, dso -> dx, dw, db, dst through partial[groups][C][W + 1]. Step: the pool is st_out
// (in place), idx/acc/first per sequence, L slots.
struct ConvParams {
  int n_seqs;
  long long T;
  int C, W, act;
  const int *cu;
  const void *x;
  const float *w, *bias;
  const void *st_in;
  void *y, *st_out;
  const void *dy;
  const float *dso;
  float *dx, *dw, *db, *dst, *partial;
  int groups;
  int L, n_slots;
  const int *idx, *acc, *first;
  int *status;
  long long prefetch_dist;   // step: CTA b brings the state and token rows of CTA b + prefetch_dist into L2
};
cudaError_t launch_conv_fwd(const ConvParams &p, bool f32, cudaStream_t s);
cudaError_t launch_conv_bwd(const ConvParams &p, bool f32, cudaStream_t s);
cudaError_t launch_conv_step(const ConvParams &p, bool f32, cudaStream_t s);
int conv_bwd_groups(long long T, int C, int W, bool f32);
cudaError_t launch_bwd_chunk_tc(const BwdChunkParams &p, cudaStream_t s);
cudaError_t launch_bwd_scan_f32(const BwdScanParams &p, cudaStream_t s);    // fp32 I/O dS scan
cudaError_t launch_bwd_chunk_f32(const BwdF32Params &p, cudaStream_t s);   // fp32 I/O chunk gradients
cudaError_t launch_step(const StepParams &p, bool f32, cudaStream_t s);
cudaError_t launch_cp_combine(int n_seqs, int n_segments, int heads, const float *M, const float *b, const float *h0,
                              float *s_in, cudaStream_t s);
// Segment offsets [N * P + 1] of P chunk-aligned segments per sequence (cu NULL: N equal sequences)
cudaError_t launch_cp_segments(const int *cu, int n_seqs, long long total, int P, int *seg, cudaStream_t s);
// hT[n] = hseg[n * P + P - 1] for the N sequences ([N][H][128][128] fp32 each)
cudaError_t launch_cp_last(const float *hseg, int n_seqs, int P, int heads, float *hT, cudaStream_t s);

// Sets the message that kda_last_error() returns on this host thread.
void set_last_error(const char *msg);

}  // namespace kda
