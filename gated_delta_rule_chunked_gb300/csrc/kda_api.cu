// kda_api.cu -- the extern "C" entry points of libkda.so (see include/kda.h).
//
// Validates every argument before anything is enqueued, carves the caller's
// workspace, and launches the kernels on the caller's stream:
//   kda_fwd:  chunk table -> chunk prep (parallel over chunks x heads)
//             -> forward state scan (sequences x heads x value slices)
//   kda_bwd:  chunk table -> reverse dS scan -> chunk gradients (one tcgen05 kernel
//             per chunk and head; the chunk records come from the forward's prep)
//   kda_step: one decode kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <string>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

thread_local std::string g_last_error;
cudaEvent_t *g_prof_events = nullptr;
int g_prof_n = 0;

void mark(int i, cudaStream_t s) {
  if (g_prof_events && i < g_prof_n) cudaEventRecord(g_prof_events[i], s);
}

kda_status fail(kda_status s, const char *fmt, const char *what = "") {
  char buf[512];
  std::snprintf(buf, sizeof buf, fmt, what);
  g_last_error = buf;
  return s;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

long long max_chunks(const kda_fwd_args *a) {
  return a->total_tokens / 64 + (long long)a->n_seqs;
}

size_t elem_size(int io) { return io == KDA_F32 ? 4 : 2; }

// Workspace carving shared by the forward and the backward.
struct WsPlan {
  size_t cu, choff, img, dsaved, aux, scratch, bytes;
};

WsPlan plan(const kda_fwd_args *a, bool bwd) {
  WsPlan w{};
  const size_t n1 = (size_t)a->n_seqs + 1;
  const size_t mc = (size_t)max_chunks(a), H = (size_t)a->heads;
  const kda::ImgLayout L((int)elem_size(a->io_dtype));
  w.cu = 0;
  w.choff = round_up(w.cu + n1 * 4, 256);
  size_t end = w.choff + n1 * 4;
  if (!bwd) {   // the forward record (the backward's records come with `saved`)
    w.img = round_up(end, 256);
    end = w.img + mc * H * (a->io_dtype == KDA_F32 ? L.bytes : (size_t)kda::TcRec::BYTES);
  } else {
    w.dsaved = round_up(end, 256);
    end = w.dsaved + mc * H * 128 * 128 * elem_size(a->io_dtype);
    if (a->io_dtype == KDA_F32) {   // the fp32 backward recomputes the records, A and T
      w.img = round_up(end, 256);
      end = w.img + mc * H * L.bytes;
      w.aux = round_up(end, 256);
      end = w.aux + mc * H * 2 * 64 * 64 * sizeof(float);
      w.scratch = round_up(end, 256);
      end = w.scratch + mc * H * kda::BWD_F32_SCRATCH * sizeof(float);
    }
  }
  w.bytes = round_up(end, 256);
  return w;
}

// TMA tensor maps (the driver's cuTensorMapEncodeTiled, reached through the runtime).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;   // a racing second lookup stores the same pointer
  if (!fn) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// Token-major [total][H][128] tensor as a 3D map (channel, head, token) with a box of
// box_c channels x 1 head x 64 tokens; 128-byte swizzle when `swz`.
bool map_tokens(CUtensorMap *m, const void *base, bool f32, long long total, int H, int box_c, bool swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t esz = f32 ? 4 : 2;
  const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)total};
  const cuuint64_t strides[2] = {128 * esz, (cuuint64_t)H * 128 * esz};
  const cuuint32_t box[3] = {(cuuint32_t)box_c, 1, 64}, estr[3] = {1, 1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The prep's fp32 {A, T} array ([items][2][64][64]) as [items * 128 rows][64], box 32 x 64 with the
// 128-byte swizzle: one box is one K-block of a K-major tf32 operand tile.
bool map_aux(CUtensorMap *m, const void *base, size_t items) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {64, (cuuint64_t)items * 128};
  const cuuint64_t strides[1] = {64 * 4};
  const cuuint32_t box[2] = {32, 64}, estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// What kda_fwd writes to `saved` for kda_bwd, per (chunk, head), as consecutive arrays:
// the chunk-start states (io type, S^T in the scans' operand-tile layout) and, for bf16,
// the forward's chunk record itself (TcRec: the dS scan and the chunk-gradient kernel read
// it MN-major where they need the transposed tiles), the fp32 A and T of the prep, and Kt.
struct SavedPlan {
  size_t states, aux, rec, kt, bytes;
};

SavedPlan saved_plan(const kda_fwd_args *a) {
  SavedPlan sp{};
  const size_t n = (size_t)max_chunks(a) * a->heads;
  sp.states = 0;
  size_t end = n * 128 * 128 * elem_size(a->io_dtype);
  if (a->io_dtype != KDA_F32) {
    sp.aux = round_up(end, 256);
    end = sp.aux + n * 2 * 64 * 64 * sizeof(float);
    sp.rec = round_up(end, 256);
    end = sp.rec + n * kda::TcRec::BYTES;
    sp.kt = round_up(end, 256);
    end = sp.kt + n * kda::KtRec::BYTES;
  }
  sp.bytes = round_up(end, 256);
  return sp;
}

kda_status check_fwd(const kda_fwd_args *a, const char *who) {
  if (!a) return fail(KDA_ERR_INVALID_ARG, "%s: args is NULL", who);
  if (a->dk != 128 || a->dv != 128 || a->chunk != 64)
    return fail(KDA_ERR_UNSUPPORTED, "%s: only dk = dv = 128 and chunk = 64 are supported", who);
  if (a->io_dtype != KDA_BF16 && a->io_dtype != KDA_F32)
    return fail(KDA_ERR_UNSUPPORTED, "%s: io_dtype must be KDA_BF16 or KDA_F32", who);
  if (a->n_seqs < 1 || a->heads < 1 || a->total_tokens < 0 || a->total_tokens > 0x7fffffffLL)
    return fail(KDA_ERR_INVALID_ARG, "%s: need n_seqs >= 1, heads >= 1, 0 <= total_tokens < 2^31", who);
  if (!a->cu_seqlens && a->total_tokens % a->n_seqs != 0)
    return fail(KDA_ERR_INVALID_ARG, "%s: without cu_seqlens total_tokens must be a multiple of n_seqs", who);
  if (a->cu_seqlens && !aligned(a->cu_seqlens, 4))
    return fail(KDA_ERR_INVALID_ARG, "%s: cu_seqlens must be 4-byte aligned", who);
  const void *need[] = {a->q, a->k, a->v, a->g, a->o};
  const char *names[] = {"q", "k", "v", "g", "o"};
  // v and o may be NULL (zero values / no output) in a forward that saves nothing
  const bool vo_optional = !a->saved;
  for (int i = 0; i < 5; ++i) {
    const bool optional = vo_optional && (i == 2 || i == 4);
    if (!need[i] && a->total_tokens > 0 && !optional)
      return fail(KDA_ERR_INVALID_ARG, "%s: required pointer is NULL", names[i]);
    if (!aligned(need[i], 16)) return fail(KDA_ERR_INVALID_ARG, "%s: pointer is not 16-byte aligned", names[i]);
  }
  if (a->skip_prep && a->saved)
    return fail(KDA_ERR_UNSUPPORTED, "%s: skip_prep needs no saved", who);
  if (!a->beta && a->total_tokens > 0) return fail(KDA_ERR_INVALID_ARG, "%s: beta is NULL", who);
  if (!aligned(a->beta, 4)) return fail(KDA_ERR_INVALID_ARG, "%s: beta is not 4-byte aligned", who);
  const void *opt[] = {a->h0, a->hT, a->saved, a->workspace};
  const char *onames[] = {"h0", "hT", "saved", "workspace"};
  for (int i = 0; i < 4; ++i)
    if (!aligned(opt[i], 16)) return fail(KDA_ERR_INVALID_ARG, "%s: pointer is not 16-byte aligned", onames[i]);
  if (a->dev_status && !aligned(a->dev_status, 4))
    return fail(KDA_ERR_INVALID_ARG, "%s: dev_status is not 4-byte aligned", who);
  if (a->wait_limit_ns < 0) return fail(KDA_ERR_INVALID_ARG, "%s: wait_limit_ns must be >= 0", who);
  if (a->debug_starve && a->io_dtype != KDA_BF16)
    return fail(KDA_ERR_UNSUPPORTED, "%s: debug_starve needs io_dtype KDA_BF16", who);
  return KDA_OK;
}

kda::SeqGeom geom(const kda_fwd_args *a, char *ws, const WsPlan &w) {
  kda::SeqGeom g;
  g.n_seqs = a->n_seqs;
  g.total = a->total_tokens;
  g.heads = a->heads;
  g.max_chunks = (int)max_chunks(a);
  g.cu = reinterpret_cast<const int *>(ws + w.cu);
  g.chunk_off = reinterpret_cast<const int *>(ws + w.choff);
  return g;
}

kda_status cuda_fail(cudaError_t e, const char *stage) {
  char buf[256];
  std::snprintf(buf, sizeof buf, "%s: %s", stage, cudaGetErrorString(e));
  g_last_error = buf;
  return KDA_ERR_CUDA;
}

int pick_slice(const kda_fwd_args *a) {
  // value-column slice per scan CTA: enough chains to cover the GPU twice
  const long long units = (long long)a->n_seqs * a->heads;
  return units * 2 >= 2LL * sm_count() ? 64 : 32;
}

}  // namespace

void kda::set_last_error(const char *msg) { g_last_error = msg ? msg : ""; }

extern "C" {

int32_t kda_abi_version(void) { return 5; }

namespace {
kda_status check_attnres(const kda_attnres_fwd_args *a, const char *who) {
  if (!a) return fail(KDA_ERR_INVALID_ARG, "%s: args is NULL", who);
  if (a->io_dtype != KDA_BF16 && a->io_dtype != KDA_F32)
    return fail(KDA_ERR_UNSUPPORTED, "%s: io_dtype must be KDA_BF16 or KDA_F32", who);
  if (a->n_sources < 1 || a->n_sources > KDA_ATTNRES_MAX_SOURCES || a->tokens < 0 || a->tokens > 0x7fffffffLL)
    return fail(KDA_ERR_INVALID_ARG, "%s: need 1 <= n_sources <= 9 and 0 <= tokens < 2^31", who);
  if (a->dim < 8 || a->dim > 16384 || a->dim % 8 != 0)
    return fail(KDA_ERR_UNSUPPORTED, "%s: dim must be a multiple of 8 in 8..16384", who);
  if (!(a->eps > 0.f)) return fail(KDA_ERR_INVALID_ARG, "%s: eps must be positive", who);
  if (a->tokens == 0) return KDA_OK;
  for (int i = 0; i < a->n_sources; ++i)
    if (!a->src[i] || !aligned(a->src[i], 16)) return fail(KDA_ERR_INVALID_ARG, "%s: a source is NULL or misaligned", who);
  if (!a->w || !aligned(a->w, 16)) return fail(KDA_ERR_INVALID_ARG, "%s: w is NULL or misaligned", who);
  if (!a->alpha || !a->rstd || !a->logit) return fail(KDA_ERR_INVALID_ARG, "%s: alpha, rstd, logit are required", who);
  return KDA_OK;
}

kda::AttnresParams attnres_params(const kda_attnres_fwd_args *a) {
  kda::AttnresParams p{};
  p.S = a->n_sources;
  p.T = a->tokens;
  p.dim = a->dim;
  p.eps = a->eps;
  for (int i = 0; i < a->n_sources; ++i) p.src[i] = a->src[i];
  p.w = a->w;
  p.out = a->out;
  p.alpha = a->alpha;
  p.rstd = a->rstd;
  p.logit = a->logit;
  return p;
}
}  // namespace

kda_status kda_attnres_fwd(const kda_attnres_fwd_args *a, cudaStream_t stream) {
  kda_status st = check_attnres(a, "kda_attnres_fwd");
  if (st != KDA_OK) return st;
  if (a->tokens == 0) {
    g_last_error.clear();
    return KDA_OK;
  }
  if (!a->out || !aligned(a->out, 16)) return fail(KDA_ERR_INVALID_ARG, "%s: out is NULL or misaligned", "kda_attnres_fwd");
  const cudaError_t e = kda::launch_attnres_fwd(attnres_params(a), a->io_dtype == KDA_F32, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_attnres_fwd");
  g_last_error.clear();
  return KDA_OK;
}

size_t kda_attnres_bwd_workspace_size(const kda_attnres_bwd_args *a) {
  if (!a || a->fwd.dim < 8 || a->fwd.dim > 16384) return 0;
  if (a->fwd.n_sources < 1 || a->fwd.n_sources > KDA_ATTNRES_MAX_SOURCES) return 0;
  return (size_t)kda::attnres_bwd_ctas(a->fwd.tokens, a->fwd.io_dtype == KDA_F32, a->fwd.dim, a->fwd.n_sources) *
         a->fwd.dim * sizeof(float);
}

kda_status kda_attnres_bwd(const kda_attnres_bwd_args *a, cudaStream_t stream) {
  if (!a) return fail(KDA_ERR_INVALID_ARG, "%s: args is NULL", "kda_attnres_bwd");
  kda_status st = check_attnres(&a->fwd, "kda_attnres_bwd");
  if (st != KDA_OK) return st;
  if (!a->dw || !aligned(a->dw, 4)) return fail(KDA_ERR_INVALID_ARG, "%s: dw is NULL or misaligned", "kda_attnres_bwd");
  const size_t need = kda_attnres_bwd_workspace_size(a);
  if (!a->workspace || a->workspace_bytes < need || !aligned(a->workspace, 16))
    return fail(KDA_ERR_INVALID_ARG, "%s: workspace missing, misaligned or smaller than kda_attnres_bwd_workspace_size()",
                "kda_attnres_bwd");
  if (a->fwd.tokens > 0) {
    if (!a->d_out || !aligned(a->d_out, 16)) return fail(KDA_ERR_INVALID_ARG, "%s: d_out is NULL or misaligned", "kda_attnres_bwd");
    for (int i = 0; i < a->fwd.n_sources; ++i)
      if (!a->d_src[i] || !aligned(a->d_src[i], 16))
        return fail(KDA_ERR_INVALID_ARG, "%s: a d_src is NULL or misaligned", "kda_attnres_bwd");
  }
  kda::AttnresParams p = attnres_params(&a->fwd);
  p.dout = a->d_out;
  for (int i = 0; i < a->fwd.n_sources; ++i) p.dsrc[i] = a->d_src[i];
  p.dw = a->dw;
  p.partial = static_cast<float *>(a->workspace);
  const cudaError_t e = kda::launch_attnres_bwd(p, a->fwd.io_dtype == KDA_F32, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_attnres_bwd");
  g_last_error.clear();
  return KDA_OK;
}

namespace {
kda_status check_conv(const kda_conv_args *a, const char *who) {
  if (!a) return fail(KDA_ERR_INVALID_ARG, "%s: args is NULL", who);
  if (a->io_dtype != KDA_BF16 && a->io_dtype != KDA_F32)
    return fail(KDA_ERR_UNSUPPORTED, "%s: io_dtype must be KDA_BF16 or KDA_F32", who);
  if (a->width < 1 || a->width > KDA_CONV_MAX_WIDTH)
    return fail(KDA_ERR_UNSUPPORTED, "%s: width must be 1..4", who);
  if (a->channels < 8 || a->channels % 8 != 0) return fail(KDA_ERR_UNSUPPORTED, "%s: channels must be a positive multiple of 8", who);
  if (a->activation != KDA_ACT_NONE && a->activation != KDA_ACT_SILU)
    return fail(KDA_ERR_INVALID_ARG, "%s: activation must be KDA_ACT_NONE or KDA_ACT_SILU", who);
  if (a->n_seqs < 0 || a->total_tokens < 0 || a->total_tokens > 0x7fffffffLL)
    return fail(KDA_ERR_INVALID_ARG, "%s: need n_seqs >= 0 and 0 <= total_tokens < 2^31", who);
  if (a->n_seqs == 0 && a->total_tokens > 0) return fail(KDA_ERR_INVALID_ARG, "%s: tokens without sequences", who);
  if (!a->cu_seqlens && a->n_seqs > 0 && a->total_tokens % a->n_seqs != 0)
    return fail(KDA_ERR_INVALID_ARG, "%s: without cu_seqlens total_tokens must divide into n_seqs equal sequences", who);
  if (a->cu_seqlens && !aligned(a->cu_seqlens, 4)) return fail(KDA_ERR_INVALID_ARG, "%s: cu_seqlens is misaligned", who);
  if (a->total_tokens > 0 && (!a->x || !aligned(a->x, 16))) return fail(KDA_ERR_INVALID_ARG, "%s: x is NULL or misaligned", who);
  if (!a->weight || !aligned(a->weight, 4)) return fail(KDA_ERR_INVALID_ARG, "%s: weight is NULL or misaligned", who);
  if (a->bias && !aligned(a->bias, 4)) return fail(KDA_ERR_INVALID_ARG, "%s: bias is misaligned", who);
  if (a->state_in && !aligned(a->state_in, 16)) return fail(KDA_ERR_INVALID_ARG, "%s: state_in is misaligned", who);
  return KDA_OK;
}

kda::ConvParams conv_params(const kda_conv_args *a) {
  kda::ConvParams p{};
  p.n_seqs = a->n_seqs;
  p.T = a->total_tokens;
  p.C = a->channels;
  p.W = a->width;
  p.act = a->activation == KDA_ACT_SILU;
  p.cu = a->cu_seqlens;
  p.x = a->x;
  p.w = a->weight;
  p.bias = a->bias;
  p.st_in = a->width > 1 ? a->state_in : nullptr;
  return p;
}

size_t conv_state_bytes(const kda_conv_args *a, size_t elem) {
  return (size_t)a->n_seqs * (a->width - 1) * a->channels * elem;
}

bool overlaps(const void *a, const void *b, size_t n) {
  const char *x = static_cast<const char *>(a), *y = static_cast<const char *>(b);
  return x && y && n && x < y + n && y < x + n;
}
}  // namespace

kda_status kda_conv_fwd(const kda_conv_args *a, cudaStream_t stream) {
  kda_status st = check_conv(a, "kda_conv_fwd");
  if (st != KDA_OK) return st;
  const bool f32 = a->io_dtype == KDA_F32;
  if (a->total_tokens > 0 && (!a->y || !aligned(a->y, 16)))
    return fail(KDA_ERR_INVALID_ARG, "%s: y is NULL or misaligned", "kda_conv_fwd");
  void *st_out = a->width > 1 ? a->state_out : nullptr;
  const size_t sbytes = conv_state_bytes(a, f32 ? 4 : 2);
  if (st_out && !aligned(st_out, 16)) return fail(KDA_ERR_INVALID_ARG, "%s: state_out is misaligned", "kda_conv_fwd");
  if (st_out && a->width > 1 && overlaps(st_out, a->state_in, sbytes))
    return fail(KDA_ERR_INVALID_ARG, "%s: state_out overlaps state_in", "kda_conv_fwd");
  cudaError_t e = cudaSuccess;
  if (a->total_tokens == 0) {   // every sequence is empty: the state passes through
    if (st_out && sbytes)
      e = a->state_in ? cudaMemcpyAsync(st_out, a->state_in, sbytes, cudaMemcpyDeviceToDevice, stream)
                      : cudaMemsetAsync(st_out, 0, sbytes, stream);
  } else {
    kda::ConvParams p = conv_params(a);
    p.y = a->y;
    p.st_out = st_out;
    e = kda::launch_conv_fwd(p, f32, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "kda_conv_fwd");
  g_last_error.clear();
  return KDA_OK;
}

size_t kda_conv_bwd_workspace_size(const kda_conv_bwd_args *a) {
  if (!a || a->fwd.width < 1 || a->fwd.width > KDA_CONV_MAX_WIDTH || a->fwd.channels < 8) return 0;
  return (size_t)kda::conv_bwd_groups(a->fwd.total_tokens, a->fwd.channels, a->fwd.width, a->fwd.io_dtype == KDA_F32) *
         a->fwd.channels * (a->fwd.width + 1) * sizeof(float);
}

kda_status kda_conv_bwd(const kda_conv_bwd_args *a, cudaStream_t stream) {
  if (!a) return fail(KDA_ERR_INVALID_ARG, "%s: args is NULL", "kda_conv_bwd");
  kda_status st = check_conv(&a->fwd, "kda_conv_bwd");
  if (st != KDA_OK) return st;
  const kda_conv_args *f = &a->fwd;
  if (f->total_tokens > 0 && (!a->dy || !aligned(a->dy, 16) || !a->dx || !aligned(a->dx, 16)))
    return fail(KDA_ERR_INVALID_ARG, "%s: dy and dx are required and 16-byte aligned", "kda_conv_bwd");
  if (!a->dweight || !aligned(a->dweight, 4)) return fail(KDA_ERR_INVALID_ARG, "%s: dweight is NULL or misaligned", "kda_conv_bwd");
  if (a->dbias && !aligned(a->dbias, 4)) return fail(KDA_ERR_INVALID_ARG, "%s: dbias is misaligned", "kda_conv_bwd");
  if ((a->d_state_out && !aligned(a->d_state_out, 16)) || (a->d_state_in && !aligned(a->d_state_in, 16)))
    return fail(KDA_ERR_INVALID_ARG, "%s: d_state_out / d_state_in misaligned", "kda_conv_bwd");
  const size_t need = kda_conv_bwd_workspace_size(a);
  if (!a->workspace || a->workspace_bytes < need || !aligned(a->workspace, 16))
    return fail(KDA_ERR_INVALID_ARG, "%s: workspace missing, misaligned or smaller than kda_conv_bwd_workspace_size()",
                "kda_conv_bwd");
  kda::ConvParams p = conv_params(f);
  p.dy = a->dy;
  p.dso = f->width > 1 ? a->d_state_out : nullptr;
  p.dx = a->dx;
  p.dw = a->dweight;
  p.db = a->dbias;
  p.dst = f->width > 1 ? a->d_state_in : nullptr;
  p.partial = static_cast<float *>(a->workspace);
  p.groups = kda::conv_bwd_groups(f->total_tokens, f->channels, f->width, f->io_dtype == KDA_F32);
  cudaError_t e = cudaSuccess;
  const size_t sbytes = conv_state_bytes(f, 4);
  if (f->total_tokens == 0 && p.dst && sbytes)   // every sequence is empty
    e = p.dso ? cudaMemcpyAsync(p.dst, p.dso, sbytes, cudaMemcpyDeviceToDevice, stream)
              : cudaMemsetAsync(p.dst, 0, sbytes, stream);
  if (e == cudaSuccess) e = kda::launch_conv_bwd(p, f->io_dtype == KDA_F32, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_conv_bwd");
  g_last_error.clear();
  return KDA_OK;
}

kda_status kda_conv_step(const kda_conv_step_args *a, cudaStream_t stream) {
  const char *who = "kda_conv_step";
  if (!a) return fail(KDA_ERR_INVALID_ARG, "%s: args is NULL", who);
  if (a->io_dtype != KDA_BF16 && a->io_dtype != KDA_F32)
    return fail(KDA_ERR_UNSUPPORTED, "%s: io_dtype must be KDA_BF16 or KDA_F32", who);
  if (a->width < 1 || a->width > KDA_CONV_MAX_WIDTH)
    return fail(KDA_ERR_UNSUPPORTED, "%s: width must be 1..4", who);
  if (a->channels < 8 || a->channels % 8 != 0) return fail(KDA_ERR_UNSUPPORTED, "%s: channels must be a positive multiple of 8", who);
  if (a->activation != KDA_ACT_NONE && a->activation != KDA_ACT_SILU)
    return fail(KDA_ERR_INVALID_ARG, "%s: activation must be KDA_ACT_NONE or KDA_ACT_SILU", who);
  if (a->n_seqs < 0 || a->n_seqs > 65535 || a->steps < 1 || a->steps > 8)
    return fail(KDA_ERR_INVALID_ARG, "%s: need 0 <= n_seqs <= 65535 and 1 <= steps <= 8", who);
  if (a->n_seqs == 0) {
    g_last_error.clear();
    return KDA_OK;
  }
  const int n_slots = a->state_indices ? a->n_slots : a->n_seqs;
  if (a->state_indices && a->n_slots < 1) return fail(KDA_ERR_INVALID_ARG, "%s: n_slots must be >= 1 with state_indices", who);
  if (!a->x || !aligned(a->x, 16) || !a->y || !aligned(a->y, 16))
    return fail(KDA_ERR_INVALID_ARG, "%s: x and y are required and 16-byte aligned", who);
  if (!a->weight || !aligned(a->weight, 4) || (a->bias && !aligned(a->bias, 4)))
    return fail(KDA_ERR_INVALID_ARG, "%s: weight is NULL or weight / bias misaligned", who);
  if (a->width > 1 && (!a->state || !aligned(a->state, 16)))
    return fail(KDA_ERR_INVALID_ARG, "%s: state is NULL or misaligned", who);
  if ((a->state_indices && !aligned(a->state_indices, 4)) || (a->accept_len && !aligned(a->accept_len, 4)) ||
      (a->first_slot && !aligned(a->first_slot, 4)) || (a->dev_status && !aligned(a->dev_status, 4)))
    return fail(KDA_ERR_INVALID_ARG, "%s: an int32 array is misaligned", who);
  kda::ConvParams p{};
  p.n_seqs = a->n_seqs;
  p.C = a->channels;
  p.W = a->width;
  p.act = a->activation == KDA_ACT_SILU;
  p.x = a->x;
  p.w = a->weight;
  p.bias = a->bias;
  p.y = a->y;
  p.st_out = a->state;
  p.L = a->steps;
  p.n_slots = n_slots;
  p.idx = a->state_indices;
  p.acc = a->accept_len;
  p.first = a->first_slot;
  p.status = a->dev_status;
  const cudaError_t e = kda::launch_conv_step(p, a->io_dtype == KDA_F32, stream);
  if (e != cudaSuccess) return cuda_fail(e, who);
  g_last_error.clear();
  return KDA_OK;
}

kda_status kda_cp_combine(const kda_cp_args *a, cudaStream_t stream) {
  if (!a) return fail(KDA_ERR_INVALID_ARG, "%s: args is NULL", "kda_cp_combine");
  if (a->dk != 128 || a->dv != 128)
    return fail(KDA_ERR_UNSUPPORTED, "%s: only dk = dv = 128 is supported", "kda_cp_combine");
  if (a->n_seqs < 0 || a->heads < 1 || a->n_segments < 1)
    return fail(KDA_ERR_INVALID_ARG, "%s: need n_seqs >= 0, heads >= 1, n_segments >= 1", "kda_cp_combine");
  if (a->n_seqs == 0) {
    g_last_error.clear();
    return KDA_OK;
  }
  if (!a->M || !a->b || !a->s_in) return fail(KDA_ERR_INVALID_ARG, "%s: M, b and s_in are required", "kda_cp_combine");
  if (!aligned(a->M, 16) || !aligned(a->b, 16) || !aligned(a->h0, 16) || !aligned(a->s_in, 16))
    return fail(KDA_ERR_INVALID_ARG, "%s: M, b, h0 and s_in must be 16-byte aligned", "kda_cp_combine");
  const cudaError_t e = kda::launch_cp_combine(a->n_seqs, a->n_segments, a->heads, a->M, a->b, a->h0, a->s_in, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_cp_combine");
  g_last_error.clear();
  return KDA_OK;
}

void kda_set_profile_events(cudaEvent_t *events, int32_t n_events) {
  g_prof_events = events;
  g_prof_n = events ? n_events : 0;
}

const char *kda_last_error(void) { return g_last_error.c_str(); }

size_t kda_fwd_workspace_size(const kda_fwd_args *a) {
  if (check_fwd(a, "kda_fwd_workspace_size") != KDA_OK) return 0;
  return plan(a, false).bytes;
}

size_t kda_saved_size(const kda_fwd_args *a) {
  if (check_fwd(a, "kda_saved_size") != KDA_OK) return 0;
  return saved_plan(a).bytes;
}

size_t kda_bwd_workspace_size(const kda_bwd_args *a) {
  if (!a) return 0;
  kda_fwd_args f = a->fwd;
  if (!f.o) f.o = a->dq;   // o is not used by the backward
  if (check_fwd(&f, "kda_bwd_workspace_size") != KDA_OK) return 0;
  return plan(&f, true).bytes;
}

namespace {
// The forward; hT_ident (bf16 I/O, no `saved`) asks for the paired scan launch, which also runs
// every sequence from the identity with zero values and writes those final states (the
// sequence's state map) to hT_ident.
kda_status fwd_impl(const kda_fwd_args *a, cudaStream_t stream, float *hT_ident) {
  kda_status st = check_fwd(a, "kda_fwd");
  if (st != KDA_OK) return st;
  const WsPlan w = plan(a, false);
  if (!a->workspace || a->workspace_bytes < w.bytes)
    return fail(KDA_ERR_INVALID_ARG, "%s: workspace missing or smaller than kda_fwd_workspace_size()", "kda_fwd");
  if (a->total_tokens == 0) {
    if (a->hT) {
      const size_t n = (size_t)a->n_seqs * a->heads * 128 * 128 * 4;
      cudaError_t e = a->h0 ? cudaMemcpyAsync(a->hT, a->h0, n, cudaMemcpyDeviceToDevice, stream)
                            : cudaMemsetAsync(a->hT, 0, n, stream);
      if (e != cudaSuccess) return cuda_fail(e, "kda_fwd");
    }
    g_last_error.clear();
    return KDA_OK;
  }
  char *ws = static_cast<char *>(a->workspace);
  const bool f32 = a->io_dtype == KDA_F32;
  CUtensorMap tm_q, tm_k, tm_g;
  if (!map_tokens(&tm_q, a->q, f32, a->total_tokens, a->heads, 128, false) ||
      !map_tokens(&tm_k, a->k, f32, a->total_tokens, a->heads, 128, false) ||
      !map_tokens(&tm_g, a->g, true, a->total_tokens, a->heads, 128, false))
    return fail(KDA_ERR_CUDA, "%s: could not encode the TMA tensor maps", "kda_fwd");
  kda::SeqGeom geo = geom(a, ws, w);
  cudaError_t e = kda::launch_chunk_table(a->cu_seqlens, a->n_seqs, a->total_tokens,
                                          reinterpret_cast<int *>(ws + w.cu), reinterpret_cast<int *>(ws + w.choff),
                                          stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_fwd chunk table");
  mark(0, stream);
  // with `saved` (a training forward) the chunk record goes there, with the backward's
  // extras (A, T, Kt); otherwise it lives in the workspace
  const SavedPlan sv = saved_plan(a);
  char *sd = static_cast<char *>(a->saved);
  const bool bwd_recs = !f32 && sd;
  char *rec = bwd_recs ? sd + sv.rec : ws + w.img;
  kda::PrepParams pp{};
  pp.geo = geo;
  pp.q = a->q;
  pp.k = a->k;
  pp.g = a->g;
  pp.beta = a->beta;
  pp.scale = a->scale;
  pp.img = rec;
  pp.aux = bwd_recs ? reinterpret_cast<float *>(sd + sv.aux) : nullptr;
  pp.tc_layout = f32 ? 0 : (bwd_recs ? 3 : 1);
  pp.img2 = bwd_recs ? sd + sv.kt : nullptr;
  pp.status = a->dev_status;
  pp.tm_q = tm_q;
  pp.tm_k = tm_k;
  pp.tm_g = tm_g;
  if (!a->skip_prep && (e = f32 ? kda::launch_prep(pp, true, stream) : kda::launch_prep_tc(pp, stream)) != cudaSuccess)
    return cuda_fail(e, "kda_fwd prep");
  mark(1, stream);
  kda::FwdScanParams sp{geo, a->v, rec, a->h0, a->o, a->hT, a->saved, a->dev_status, a->h0_identity != 0, {},
                        a->wait_limit_ns > 0 ? (unsigned long long)a->wait_limit_ns : 2000000000ull,
                        a->debug_starve != 0, f32 || a->saved ? nullptr : hT_ident};
  if (!f32 && a->v && !map_tokens(&sp.tm_v, a->v, false, a->total_tokens, a->heads, 64, true))
    return fail(KDA_ERR_CUDA, "%s: could not encode the TMA tensor maps", "kda_fwd");
  e = f32 ? kda::launch_fwd_scan(sp, true, pick_slice(a), stream) : kda::launch_fwd_scan_tc(sp, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_fwd scan");
  mark(2, stream);
  g_last_error.clear();
  return KDA_OK;
}
}  // namespace

kda_status kda_fwd(const kda_fwd_args *a, cudaStream_t stream) { return fwd_impl(a, stream, nullptr); }

namespace {
// fp32 I/O: the prep runs again into the workspace (records, A, T), then the fp32 dS scan and
// the two fp32 chunk kernels (kda_bwd_f32.cu). `saved` holds the chunk-start states only.
kda_status bwd_f32(const kda_bwd_args *a, const WsPlan &w, cudaStream_t stream) {
  const kda_fwd_args *f = &a->fwd;
  char *ws = static_cast<char *>(a->workspace);
  const long long T = f->total_tokens;
  CUtensorMap tm_q, tm_k, tm_g;
  if (!map_tokens(&tm_q, f->q, true, T, f->heads, 128, false) || !map_tokens(&tm_k, f->k, true, T, f->heads, 128, false) ||
      !map_tokens(&tm_g, f->g, true, T, f->heads, 128, false))
    return fail(KDA_ERR_CUDA, "%s: could not encode the TMA tensor maps", "kda_bwd");
  kda::SeqGeom geo = geom(f, ws, w);
  cudaError_t e = kda::launch_chunk_table(f->cu_seqlens, f->n_seqs, T, reinterpret_cast<int *>(ws + w.cu),
                                          reinterpret_cast<int *>(ws + w.choff), stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_bwd chunk table");
  mark(0, stream);
  kda::PrepParams pp{};
  pp.geo = geo;
  pp.q = f->q;
  pp.k = f->k;
  pp.g = f->g;
  pp.beta = f->beta;
  pp.scale = f->scale;
  pp.img = ws + w.img;
  pp.aux = reinterpret_cast<float *>(ws + w.aux);
  pp.status = f->dev_status;
  pp.tm_q = tm_q;
  pp.tm_k = tm_k;
  pp.tm_g = tm_g;
  if ((e = kda::launch_prep(pp, true, stream)) != cudaSuccess) return cuda_fail(e, "kda_bwd prep");
  kda::BwdScanParams bp{geo, a->dO, ws + w.img, a->dhT, a->dv, a->dh0, ws + w.dsaved, f->dev_status, {}};
  if ((e = kda::launch_bwd_scan_f32(bp, stream)) != cudaSuccess) return cuda_fail(e, "kda_bwd dS scan");
  mark(1, stream);
  kda::BwdF32Params cp{};
  cp.geo = geo;
  cp.q = static_cast<const float *>(f->q);
  cp.k = static_cast<const float *>(f->k);
  cp.v = static_cast<const float *>(f->v);
  cp.dO = static_cast<const float *>(a->dO);
  cp.g = f->g;
  cp.beta = f->beta;
  cp.scale = f->scale;
  cp.img = ws + w.img;
  cp.aux = reinterpret_cast<const float *>(ws + w.aux);
  cp.saved = static_cast<const float *>(f->saved);
  cp.dsaved = reinterpret_cast<const float *>(ws + w.dsaved);
  cp.dq = a->dq;
  cp.dk = a->dk;
  cp.dg = a->dg;
  cp.dbeta = a->dbeta;
  cp.scratch = reinterpret_cast<float *>(ws + w.scratch);
  cp.status = f->dev_status;
  if ((e = kda::launch_bwd_chunk_f32(cp, stream)) != cudaSuccess) return cuda_fail(e, "kda_bwd chunk grads");
  mark(2, stream);
  g_last_error.clear();
  return KDA_OK;
}
}  // namespace

kda_status kda_bwd(const kda_bwd_args *a, cudaStream_t stream) {
  if (!a) return fail(KDA_ERR_INVALID_ARG, "%s: args is NULL", "kda_bwd");
  const kda_fwd_args *f = &a->fwd;
  kda_fwd_args fcheck = *f;
  if (!fcheck.o) fcheck.o = a->dq;   // o is not used by the backward
  kda_status st = check_fwd(&fcheck, "kda_bwd");
  if (st != KDA_OK) return st;
  if (!f->v && f->total_tokens > 0) return fail(KDA_ERR_INVALID_ARG, "%s: v is NULL", "kda_bwd");
  const WsPlan w = plan(f, true);
  if (!a->workspace || a->workspace_bytes < w.bytes)
    return fail(KDA_ERR_INVALID_ARG, "%s: workspace missing or smaller than kda_bwd_workspace_size()", "kda_bwd");
  const void *need[] = {a->dO, a->dq, a->dk, a->dv, a->dg, f->saved};
  const char *names[] = {"dO", "dq", "dk", "dv", "dg", "fwd.saved"};
  for (int i = 0; i < 6; ++i) {
    if (!need[i] && f->total_tokens > 0) return fail(KDA_ERR_INVALID_ARG, "kda_bwd: %s is NULL", names[i]);
    if (!aligned(need[i], 16)) return fail(KDA_ERR_INVALID_ARG, "kda_bwd: %s is not 16-byte aligned", names[i]);
  }
  if ((!a->dbeta && f->total_tokens > 0) || !aligned(a->dbeta, 4))
    return fail(KDA_ERR_INVALID_ARG, "%s: dbeta is NULL or not 4-byte aligned", "kda_bwd");
  if (!aligned(a->dhT, 16) || !aligned(a->dh0, 16) || !aligned(a->workspace, 16))
    return fail(KDA_ERR_INVALID_ARG, "%s: dhT, dh0 or workspace is not 16-byte aligned", "kda_bwd");
  if (f->total_tokens == 0) {
    if (a->dh0) {
      const size_t n = (size_t)f->n_seqs * f->heads * 128 * 128 * 4;
      cudaError_t e = a->dhT ? cudaMemcpyAsync(a->dh0, a->dhT, n, cudaMemcpyDeviceToDevice, stream)
                             : cudaMemsetAsync(a->dh0, 0, n, stream);
      if (e != cudaSuccess) return cuda_fail(e, "kda_bwd");
    }
    g_last_error.clear();
    return KDA_OK;
  }
  char *ws = static_cast<char *>(a->workspace);
  if (f->io_dtype == KDA_F32) return bwd_f32(a, w, stream);
  // the chunk records were written by the forward's prep into `saved`
  const SavedPlan sv = saved_plan(f);
  char *sd = static_cast<char *>(f->saved);
  kda::BwdChunkParams cp{};
  const long long T = f->total_tokens;
  if (!map_tokens(&cp.tm_q, f->q, false, T, f->heads, 128, false) ||
      !map_tokens(&cp.tm_k, f->k, false, T, f->heads, 128, false) ||
      !map_tokens(&cp.tm_v, f->v, false, T, f->heads, 128, false) ||
      !map_tokens(&cp.tm_do, a->dO, false, T, f->heads, 64, true) ||
      !map_aux(&cp.tm_aux, sd + sv.aux, (size_t)max_chunks(f) * f->heads))
    return fail(KDA_ERR_CUDA, "%s: could not encode the TMA tensor maps", "kda_bwd");
  kda::SeqGeom geo = geom(f, ws, w);
  cudaError_t e = kda::launch_chunk_table(f->cu_seqlens, f->n_seqs, f->total_tokens,
                                          reinterpret_cast<int *>(ws + w.cu), reinterpret_cast<int *>(ws + w.choff),
                                          stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_bwd chunk table");
  mark(0, stream);
  kda::BwdScanParams bp{geo, a->dO, sd + sv.rec, a->dhT, a->dv, a->dh0, ws + w.dsaved, f->dev_status, cp.tm_do};
  if ((e = kda::launch_bwd_scan_tc(bp, stream)) != cudaSuccess) return cuda_fail(e, "kda_bwd dS scan");
  mark(1, stream);
  cp.geo = geo;
  cp.q = f->q;
  cp.k = f->k;
  cp.v = f->v;
  cp.dO = a->dO;
  cp.g = f->g;
  cp.beta = f->beta;
  cp.scale = f->scale;
  cp.img = sd + sv.rec;
  cp.kt = sd + sv.kt;
  cp.saved = sd + sv.states;
  cp.dsaved = ws + w.dsaved;
  cp.aux = reinterpret_cast<const float *>(sd + sv.aux);
  cp.dq = a->dq;
  cp.dk = a->dk;
  cp.dg = a->dg;
  cp.dbeta = a->dbeta;
  cp.status = f->dev_status;
  if ((e = kda::launch_bwd_chunk_tc(cp, stream)) != cudaSuccess) return cuda_fail(e, "kda_bwd chunk grads");
  mark(2, stream);
  g_last_error.clear();
  return KDA_OK;
}

namespace {
// Workspace of kda_fwd_cp: the segment table, the workspace of the segmented forward
// (N * P sequences), and three [N * P][H][128][128] fp32 state arrays (M, b, S_in; the
// last pass writes the segments' final states over M).
struct CpPlan {
  size_t seg, fws, M, b, s_in, bytes, fws_bytes;
};

CpPlan cp_plan(const kda_fwd_cp_args *c) {
  CpPlan w{};
  kda_fwd_args f = c->fwd;
  f.n_seqs = c->fwd.n_seqs * c->n_segments;
  const size_t nseg = (size_t)f.n_seqs;
  w.seg = 0;
  w.fws = round_up((nseg + 1) * 4, 256);
  w.fws_bytes = plan(&f, false).bytes;
  const size_t st = nseg * (size_t)c->fwd.heads * 128 * 128 * sizeof(float);
  w.M = round_up(w.fws + w.fws_bytes, 256);
  w.b = w.M + st;
  w.s_in = w.b + st;
  w.bytes = w.s_in + st;
  return w;
}

kda_status check_cp(const kda_fwd_cp_args *c, const char *who) {
  if (!c) return fail(KDA_ERR_INVALID_ARG, "%s: args is NULL", who);
  kda_fwd_args f = c->fwd;   // fwd.workspace is ignored (this call takes its own)
  f.workspace = nullptr;
  f.workspace_bytes = 0;
  kda_status st = check_fwd(&f, who);
  if (st != KDA_OK) return st;
  if (c->fwd.saved || c->fwd.h0_identity || c->fwd.skip_prep || c->fwd.debug_starve)
    return fail(KDA_ERR_UNSUPPORTED, "%s: needs no saved and h0_identity = skip_prep = debug_starve = 0", who);
  if (c->n_segments < 1 || (long long)c->n_segments * c->fwd.n_seqs > 0x7fffffffLL / 64)
    return fail(KDA_ERR_INVALID_ARG, "%s: need n_segments >= 1 (and n_seqs * n_segments < 2^25)", who);
  if (c->fwd.total_tokens > 0 && (!c->fwd.v || !c->fwd.o))
    return fail(KDA_ERR_INVALID_ARG, "%s: v and o are required", who);
  return KDA_OK;
}
}  // namespace

size_t kda_fwd_cp_workspace_size(const kda_fwd_cp_args *c) {
  if (check_cp(c, "kda_fwd_cp_workspace_size") != KDA_OK) return 0;
  return cp_plan(c).bytes;
}

kda_status kda_fwd_cp(const kda_fwd_cp_args *c, cudaStream_t stream) {
  kda_status st = check_cp(c, "kda_fwd_cp");
  if (st != KDA_OK) return st;
  const CpPlan w = cp_plan(c);
  if (!c->workspace || c->workspace_bytes < w.bytes || !aligned(c->workspace, 16))
    return fail(KDA_ERR_INVALID_ARG, "%s: workspace missing, misaligned or smaller than kda_fwd_cp_workspace_size()",
                "kda_fwd_cp");
  const kda_fwd_args &f = c->fwd;
  const int N = f.n_seqs, P = c->n_segments, H = f.heads;
  if (f.total_tokens == 0) {   // every segment empty: hT = h0
    if (f.hT) {
      const size_t n = (size_t)N * H * 128 * 128 * 4;
      cudaError_t e = f.h0 ? cudaMemcpyAsync(f.hT, f.h0, n, cudaMemcpyDeviceToDevice, stream)
                           : cudaMemsetAsync(f.hT, 0, n, stream);
      if (e != cudaSuccess) return cuda_fail(e, "kda_fwd_cp");
    }
    g_last_error.clear();
    return KDA_OK;
  }
  char *ws = static_cast<char *>(c->workspace);
  int *seg = reinterpret_cast<int *>(ws + w.seg);
  float *M = reinterpret_cast<float *>(ws + w.M), *b = reinterpret_cast<float *>(ws + w.b);
  float *s_in = reinterpret_cast<float *>(ws + w.s_in);
  cudaError_t e = kda::launch_cp_segments(f.cu_seqlens, N, f.total_tokens, P, seg, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_fwd_cp segments");
  // the segmented problem: N * P sequences with the segment table as offsets
  kda_fwd_args s = f;
  s.n_seqs = N * P;
  s.cu_seqlens = seg;
  s.workspace = ws + w.fws;
  s.workspace_bytes = w.fws_bytes;
  if (f.io_dtype != KDA_F32) {
    // passes 1 and 2 in one launch: the chunk records, then paired scans per (segment, head), one
    // for the segment maps M (identity start, zero values), one for the offsets b (zero start)
    kda_fwd_args p12 = s;
    p12.o = nullptr;
    p12.h0 = nullptr;
    p12.hT = b;
    if ((st = fwd_impl(&p12, stream, M)) != KDA_OK) return st;
  } else {
    // pass 1: chunk records and the segment maps M (identity start, zero values, no outputs)
    kda_fwd_args p1 = s;
    p1.v = nullptr;
    p1.o = nullptr;
    p1.h0 = nullptr;
    p1.hT = M;
    p1.h0_identity = 1;
    if ((st = kda_fwd(&p1, stream)) != KDA_OK) return st;
    // pass 2: the segment offsets b (zero start, same records)
    kda_fwd_args p2 = s;
    p2.o = nullptr;
    p2.h0 = nullptr;
    p2.hT = b;
    p2.skip_prep = 1;
    if ((st = kda_fwd(&p2, stream)) != KDA_OK) return st;
  }
  // combine: the state entering each segment
  if ((e = kda::launch_cp_combine(N, P, H, M, b, f.h0, s_in, stream)) != cudaSuccess)
    return cuda_fail(e, "kda_fwd_cp combine");
  // pass 3: every segment from its entering state; its final states land over M
  kda_fwd_args p3 = s;
  p3.h0 = s_in;
  p3.hT = M;
  p3.skip_prep = 1;
  if ((st = kda_fwd(&p3, stream)) != KDA_OK) return st;
  if (f.hT && (e = kda::launch_cp_last(M, N, P, H, f.hT, stream)) != cudaSuccess)
    return cuda_fail(e, "kda_fwd_cp final states");
  g_last_error.clear();
  return KDA_OK;
}

kda_status kda_step(const kda_step_args *a, cudaStream_t stream) {
  if (!a) return fail(KDA_ERR_INVALID_ARG, "%s: args is NULL", "kda_step");
  if (a->dk != 128 || a->dv != 128) return fail(KDA_ERR_UNSUPPORTED, "%s: only dk = dv = 128 is supported", "kda_step");
  if (a->io_dtype != KDA_BF16 && a->io_dtype != KDA_F32)
    return fail(KDA_ERR_UNSUPPORTED, "%s: io_dtype must be KDA_BF16 or KDA_F32", "kda_step");
  if (a->n_seqs < 0 || a->heads < 1 || a->steps < 1 || a->steps > 8)
    return fail(KDA_ERR_INVALID_ARG, "%s: need n_seqs >= 0, heads >= 1, 1 <= steps <= 8", "kda_step");
  if (a->n_seqs == 0) {
    g_last_error.clear();
    return KDA_OK;
  }
  const void *need[] = {a->q, a->k, a->v, a->g, a->state, a->o};
  const char *names[] = {"q", "k", "v", "g", "state", "o"};
  for (int i = 0; i < 6; ++i) {
    if (!need[i]) return fail(KDA_ERR_INVALID_ARG, "kda_step: %s is NULL", names[i]);
    if (!aligned(need[i], 16)) return fail(KDA_ERR_INVALID_ARG, "kda_step: %s is not 16-byte aligned", names[i]);
  }
  if (!a->beta || !aligned(a->beta, 4)) return fail(KDA_ERR_INVALID_ARG, "%s: beta is NULL or misaligned", "kda_step");
  if (!aligned(a->accept_len, 4) || !aligned(a->state_indices, 4) || !aligned(a->first_slot, 4) ||
      !aligned(a->dev_status, 4))
    return fail(KDA_ERR_INVALID_ARG, "%s: accept_len, state_indices, first_slot or dev_status is misaligned",
                "kda_step");
  if (a->state_indices && a->n_slots < 1)
    return fail(KDA_ERR_INVALID_ARG, "%s: state_indices needs n_slots >= 1", "kda_step");
  kda::StepParams p{a->n_seqs, a->steps, a->heads, a->scale, a->q, a->k, a->v, a->beta, a->g, a->state,
                    a->accept_len, a->o, a->state_indices, a->n_slots, a->first_slot, a->dev_status};
  cudaError_t e = kda::launch_step(p, a->io_dtype == KDA_F32, stream);
  if (e != cudaSuccess) return cuda_fail(e, "kda_step");
  mark(0, stream);
  g_last_error.clear();
  return KDA_OK;
}

}  // extern "C"
