/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention library (libkda.so).
 *
 * Kimi Delta Attention (KDA) is linear attention whose per-head recurrent state
 * is updated with channel-wise gating ("Kimi K3 on Fireworks: Fast RL at frontier
 * scale", training section, KDA paragraph; the first page's section
 * "KDA：从循环记忆到高效 GPU 执行", whose benchmark caption counts the Q/K
 * normalisation and the gate scan as part of the KDA core). Per head, with the
 * state S of shape [dk][dv] (row c = key channel, column j = value channel):
 *
 *     q^ = scale * q / sqrt(|q|^2 + 1e-6),     k^ = k / sqrt(|k|^2 + 1e-6)
 *     S_t = (I - beta_t k^_t k^_t^T) Diag(exp(g_t)) S_{t-1} + beta_t k^_t v_t^T
 *     o_t = S_t^T q^_t
 *
 * g is the per-channel log-decay (g <= 0), beta the per-token write strength.
 * The model shape of interest is 96 heads x 128 dims with a 128 x 128 state per
 * head (architecture figure of "Kimi K3 模型结构（10）：RL 与服务中的状态管理").
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or synchronises. Every call only enqueues work on
 *    `stream` and returns; results are valid once the stream reaches that point.
 *  - Layouts are dense row-major with the listed shapes. Token-major tensors pack
 *    all sequences back to back: token t of sequence i is row cu_seqlens[i] + t.
 *  - Supported sizes: dk = dv = 128, chunk = 64, heads >= 1. Other values return
 *    KDA_ERR_UNSUPPORTED.
 *  - Tensor, state and workspace pointers must be 16-byte aligned; the int32 and
 *    per-token scalar arrays (cu_seqlens, beta, dbeta, accept_len, dev_status)
 *    need 4-byte alignment. A required pointer that is NULL or misaligned, or a
 *    workspace smaller than the matching *_workspace_size(), returns
 *    KDA_ERR_INVALID_ARG. Validation happens before any launch: on an error
 *    nothing is written.
 *  - KDA_ERR_CUDA means a launch failed (see kda_last_error()).
 *  - If dev_status is not NULL it must point to one device int32 that the caller
 *    zeroes; a kernel that gives up a bounded wait writes KDA_ERR_TIMEOUT there.
 *  - Results are deterministic: identical inputs give bit-identical outputs
 *    (no floating-point atomics anywhere).
 *  - Preconditions that are not checked: inputs are finite; g <= 0; the sum of g
 *    over any 16 consecutive tokens of one channel inside a 64-token chunk is
 *    >= -80 (every g >= -5 is enough), which keeps every gating factor in range.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,   /* NULL / misaligned pointer, bad size, small workspace */
    KDA_ERR_UNSUPPORTED = 2,   /* dk, dv, chunk or dtype outside the supported set       */
    KDA_ERR_CUDA = 3,          /* a CUDA launch failed                                   */
    KDA_ERR_TIMEOUT = 4        /* written to *dev_status by a kernel whose wait gave up  */
} kda_status;

typedef enum {
    KDA_BF16 = 0,              /* q, k, v, o, dO stored as bfloat16                     */
    KDA_F32 = 1                /* ... stored as float32                                  */
} kda_dtype;

/* Chunked training forward. */
typedef struct {
    int32_t n_seqs;            /* N >= 1 sequences                                       */
    int64_t total_tokens;      /* sum of the sequence lengths (0 allowed: no work)      */
    int32_t heads;             /* H                                                      */
    int32_t dk, dv;            /* 128, 128                                               */
    int32_t chunk;             /* 64                                                     */
    float scale;               /* multiplies q^ (1.0 for plain KDA)                      */
    int32_t io_dtype;          /* kda_dtype of q, k, v, o                                */
    const int32_t *cu_seqlens; /* [N+1] sequence offsets, cu[0]=0, cu[N]=total, or NULL:
                                  N sequences of equal length total/N                   */
    const void *q;             /* [total, H, dk]                                         */
    const void *k;             /* [total, H, dk]                                         */
    const void *v;             /* [total, H, dv], or NULL for zero values (a forward
                                  without `saved`)                                        */
    const float *beta;         /* [total, H]                                             */
    const float *g;            /* [total, H, dk] log-decay                               */
    const float *h0;           /* [N, H, dk, dv] initial states, or NULL for zero        */
    void *o;                   /* out [total, H, dv], or NULL: not written (a forward
                                  without `saved`)                                        */
    float *hT;                 /* out [N, H, dk, dv] final states, or NULL               */
    void *saved;               /* out, kda_saved_size() bytes: what kda_bwd needs from this
                                  forward (chunk-start states; for bf16 also the forward's
                                  chunk records and the prep's A, T and Kt tiles, computed
                                  in the same pass), or NULL when no backward follows     */
    void *workspace;           /* scratch, kda_fwd_workspace_size() bytes                */
    size_t workspace_bytes;
    int32_t *dev_status;       /* optional device int32, see above                       */
    /* ABI version 3: */
    int32_t h0_identity;       /* nonzero: every sequence starts from the identity state
                                  (dk = dv), h0 is ignored. With v = NULL the final state
                                  is then the sequence's linear map on its initial state  */
    int32_t skip_prep;         /* nonzero: the workspace still holds the chunk records of a
                                  previous kda_fwd (without saved, same io_dtype) on the
                                  same q, k, g, beta and sequence layout; only the scan
                                  runs (the records do not depend on v, h0 or the initial
                                  state)                                                  */
    /* ABI version 5: testing aids for the bounded waits of the bf16 state scan (leave 0) */
    int64_t wait_limit_ns;     /* limit of every bounded wait in the bf16 state scan, in ns;
                                  0 = the default of about 2 s                            */
    int32_t debug_starve;      /* nonzero (bf16 only): the scan's first CTA (sequence 0,
                                  head 0) issues none of its first copies, so its waits
                                  run out after wait_limit_ns; it writes KDA_ERR_TIMEOUT to
                                  *dev_status, leaves that head's o and hT unwritten and
                                  exits with nothing in flight. Nothing faults or hangs;
                                  the context stays usable                                */
} kda_fwd_args;

/* Backward of kda_fwd: gradients of <dO, o> + <dhT, hT>. */
typedef struct {
    kda_fwd_args fwd;          /* the forward's arguments; fwd.o, fwd.hT are ignored and
                                  fwd.saved must hold what that forward wrote             */
    const void *dO;            /* [total, H, dv] in io_dtype                             */
    const float *dhT;          /* [N, H, dk, dv] or NULL for zero                        */
    float *dq;                 /* out [total, H, dk] fp32                                */
    float *dk;                 /* out [total, H, dk] fp32                                */
    float *dv;                 /* out [total, H, dv] fp32                                */
    float *dbeta;              /* out [total, H] fp32                                    */
    float *dg;                 /* out [total, H, dk] fp32                                */
    float *dh0;                /* out [N, H, dk, dv] fp32, or NULL                       */
    void *workspace;           /* scratch, kda_bwd_workspace_size() bytes                */
    size_t workspace_bytes;
} kda_bwd_args;

/* Decode / draft-verify step: L tokens per sequence against a committed state. */
typedef struct {
    int32_t n_seqs;            /* N                                                      */
    int32_t steps;             /* L, 1..8 tokens per sequence in this call               */
    int32_t heads;             /* H                                                      */
    int32_t dk, dv;            /* 128, 128                                               */
    float scale;
    int32_t io_dtype;          /* kda_dtype of q, k, v, o                                */
    const void *q;             /* [N, L, H, dk]                                          */
    const void *k;             /* [N, L, H, dk]                                          */
    const void *v;             /* [N, L, H, dv]                                          */
    const float *beta;         /* [N, L, H]                                              */
    const float *g;            /* [N, L, H, dk]                                          */
    float *state;              /* in/out [N, H, dk, dv] (or [P, H, dk, dv] with state_indices):
                                  read, then overwritten with the state after accept_len[i]
                                  token slots (untouched if 0)                            */
    const int32_t *accept_len; /* [N] in 0..L, or NULL meaning L for every sequence      */
    void *o;                   /* out [N, L, H, dv]: outputs of the L token slots (slots
                                  before first_slot[i] are not written)                   */
    /* ABI version 2: */
    const int32_t *state_indices; /* [N] slot of sequence i in a pool of n_slots states, or
                                     NULL (slot i); distinct slots for sequences that
                                     commit. A slot outside 0..n_slots-1 leaves that
                                     sequence untouched and writes KDA_ERR_INVALID_ARG to
                                     *dev_status                                          */
    int32_t n_slots;              /* P, the pool size (used with state_indices)           */
    const int32_t *first_slot;    /* [N] in 0..L: slots before first_slot[i] are padding,
                                     exact identities (no state change, no output), or
                                     NULL (0)                                             */
    int32_t *dev_status;          /* optional device int32, as in kda_fwd_args            */
} kda_step_args;

/*
 * kda_fwd -- chunked forward (chunk 64). Per chunk the intra-chunk work (gated
 * k.k^T / q.k^T blocks, the WY/UT triangular solve) runs in parallel over all
 * chunks and heads, and a sequential scan passes the 128x128 state between
 * chunks (the KDA paragraph: chunk-local work in parallel, little state between).
 */
kda_status kda_fwd(const kda_fwd_args *args, cudaStream_t stream);
size_t kda_fwd_workspace_size(const kda_fwd_args *args);
/* Bytes that kda_fwd writes to args->saved for kda_bwd: per (chunk, head) the
 * chunk-start state (io type) and, for bf16 I/O, the forward's chunk record with the
 * prep's A, T and Kt tiles (about 113 KB more per chunk and head). */
size_t kda_saved_size(const kda_fwd_args *args);

/* kda_bwd -- gradients for q, k, v, beta, g and the initial state (the pages
 * report a matching backward kernel next to the forward one). `fwd.saved` is the
 * buffer a kda_fwd with the same inputs filled. bf16 I/O runs on the tensor cores
 * (bf16 operands, fp32 accumulation; within 1e-2 of the exact gradients); fp32 I/O
 * forms every product in fp32 on the CUDA cores (within 1e-4) and recomputes the
 * chunk records, A and T in its workspace, which is therefore larger: about 260 KB
 * per (chunk, head) against 32 KB for bf16. */
kda_status kda_bwd(const kda_bwd_args *args, cudaStream_t stream);
size_t kda_bwd_workspace_size(const kda_bwd_args *args);

/* kda_step -- recurrent decode over L <= 8 tokens, returning all L outputs and
 * committing the state only through the accepted prefix, as ReplaySSM advances
 * KDA state only through accepted tokens ("Kimi K3 on Fireworks", rollout
 * section, speculative decoding paragraph). Needs no workspace.
 *
 * Two-phase use (verify, then replay): a verify call runs the draft tokens with
 * accept_len = 0, so the committed state is not written. Once a_i of them are
 * accepted, the next call replays those a_i tokens and verifies the next draft in
 * one pass: its slots hold [R - a_i padding | the a_i accepted tokens | the new
 * draft], with first_slot[i] = R - a_i and accept_len[i] = R, so the committed
 * state advances exactly through the accepted tokens and the outputs of the new
 * draft are computed from it. state_indices addresses states in a pool (paged
 * state cache), so sequences keep their slot across calls. */
kda_status kda_step(const kda_step_args *args, cudaStream_t stream);

/*
 * kda_cp_combine -- context parallelism by segment-affine combine (the pages' CP
 * paragraphs: the sequence split across devices, with a state exchange between them).
 * Each sequence is split into P consecutive segments; a segment maps its incoming
 * state affinely, S_out = M S_in + b, where M (dk x dk) is the final state of a forward
 * over the segment from the identity with zero values (h0_identity, v = NULL) and b is
 * the final state of a forward from zero. Given M and b of every segment (computed
 * independently, e.g. on P devices), this writes the state entering each segment:
 * S_in[0] = h0, S_in[k+1] = M[k] S_in[k] + b[k]; a forward over each segment from
 * S_in then reproduces the unsplit forward.
 */
typedef struct {
    int32_t n_seqs;            /* N                                                      */
    int32_t n_segments;        /* P >= 1 segments per sequence                           */
    int32_t heads;             /* H                                                      */
    int32_t dk, dv;            /* 128, 128                                               */
    const float *M;            /* [N, P, H, dk, dk] fp32                                 */
    const float *b;            /* [N, P, H, dk, dv] fp32                                 */
    const float *h0;           /* [N, H, dk, dv] fp32, or NULL for zero                  */
    float *s_in;               /* out [N, P, H, dk, dv] fp32                             */
} kda_cp_args;

kda_status kda_cp_combine(const kda_cp_args *args, cudaStream_t stream);

/*
 * kda_fwd_cp -- the whole context-parallel forward on one device: each sequence of
 * args->fwd is cut into n_segments consecutive runs of whole 64-token chunks (as
 * equal as chunk alignment allows; trailing segments of a short sequence may be
 * empty), and the segments are processed as independent sequences the way P devices
 * would process their own segment ("Kimi K3 on Fireworks", training section, CP
 * bullet: contiguous token ranges kept for KDA's recurrent state propagation):
 *   1. the chunk records of every segment (they depend on q, k, g, beta only);
 *   2. each segment's map M: final state from the identity with zero values;
 *   3. each segment's offset b: final state from zero (with bf16 I/O, 2 and 3 run as one
 *      launch, the two scans of a segment side by side);
 *   4. kda_cp_combine: the state entering each segment;
 *   5. a forward over every segment from its entering state, writing o, and the
 *      final state of each sequence's last segment to hT.
 * The result equals kda_fwd on args->fwd up to rounding. Everything is enqueued on
 * `stream`; nothing is copied to the host. Supported: io_dtype KDA_BF16 or KDA_F32 (fp32
 * products throughout, like kda_fwd), saved = NULL, h0_identity = skip_prep = 0 (the
 * other kda_fwd_args fields as for kda_fwd; fwd.workspace is ignored: this call takes
 * its own).
 */
typedef struct {
    kda_fwd_args fwd;          /* the unsplit forward (o required, hT optional)           */
    int32_t n_segments;        /* P >= 1                                                  */
    void *workspace;           /* kda_fwd_cp_workspace_size() bytes: segment table,
                                  records, and the M, b and entering states of the
                                  N * P segments (3 x 64 KiB per segment and head)         */
    size_t workspace_bytes;
} kda_fwd_cp_args;

kda_status kda_fwd_cp(const kda_fwd_cp_args *args, cudaStream_t stream);
size_t kda_fwd_cp_workspace_size(const kda_fwd_cp_args *args);

/*
 * Attention Residuals ("Kimi K3 on Fireworks", training section, Attention Residuals
 * paragraph; the second page's model figure): a sublayer combines up to 9 earlier
 * representations of each token (the embedding, finished blocks, the current block's
 * partial sum) with softmax weights scored by a learned pseudo-query w:
 *     r_i = (mean_c x_ic^2 + eps)^(-1/2),   logit_i = r_i (w . x_i),
 *     alpha = softmax_i(logit),              out = sum_i alpha_i x_i.
 * One fused pass per token: the normalised sources and weights are never stored
 * beyond three [T, S] fp32 statistics for the backward.
 */
#define KDA_ATTNRES_MAX_SOURCES 9

typedef struct {
    int32_t n_sources;         /* S, 1..9                                                */
    int64_t tokens;            /* T                                                      */
    int32_t dim;               /* d, a multiple of 8, at most 16384                      */
    float eps;                 /* inside the RMS (1e-6 in the tests)                     */
    int32_t io_dtype;          /* kda_dtype of the sources, out, d_out, d_src            */
    const void *src[KDA_ATTNRES_MAX_SOURCES];   /* S tensors [T, d]                     */
    const float *w;            /* [d] pseudo-query                                       */
    void *out;                 /* out [T, d]                                             */
    float *alpha;              /* out [T, S] softmax weights   (kept for the backward)   */
    float *rstd;               /* out [T, S] r_i               (kept for the backward)   */
    float *logit;              /* out [T, S] logit_i           (kept for the backward)   */
} kda_attnres_fwd_args;

typedef struct {
    kda_attnres_fwd_args fwd;  /* the forward's arguments and statistics (out unused)    */
    const void *d_out;         /* [T, d]                                                 */
    void *d_src[KDA_ATTNRES_MAX_SOURCES];       /* out, S tensors [T, d]               */
    float *dw;                 /* out [d] fp32                                           */
    void *workspace;           /* kda_attnres_bwd_workspace_size() bytes (dw partials)   */
    size_t workspace_bytes;
} kda_attnres_bwd_args;

kda_status kda_attnres_fwd(const kda_attnres_fwd_args *args, cudaStream_t stream);
kda_status kda_attnres_bwd(const kda_attnres_bwd_args *args, cudaStream_t stream);
size_t kda_attnres_bwd_workspace_size(const kda_attnres_bwd_args *args);

/*
 * Short convolution on the KDA input side ("Kimi K3 on Fireworks: Fast RL at frontier
 * scale", rollout section, the paragraph on inline versus disaggregated serving, and its
 * translation under "选择内联或分离式rollout服务" in "Fireworks 发布 Kimi K3 大规模强化学习
 * 技术报告": a sequence handed to another pool carries its KDA recurrent state together
 * with its convolution state). The pages name the convolution state and nothing else;
 * this library reads it as a causal
 * depthwise 1-D convolution of width W over the token axis, one filter per channel, with
 * an optional bias and SiLU, applied to the q, k, v projections before the KDA core:
 *     z[t, c] = bias[c] + sum_{j < W} weight[c, j] * x[t - (W - 1) + j, c]
 *     y[t, c] = act(z[t, c]),   act = identity or SiLU (z / (1 + e^-z))
 * Positions before a sequence's first token read its convolution state: the W - 1 inputs
 * that preceded it, oldest first (state[n, i, :] is position i - (W - 1)); NULL reads as
 * zeros. The state after a sequence is its last W - 1 inputs in the same layout (taken
 * partly from the incoming state when the sequence is shorter than W - 1). Channels are
 * independent, so x may be one projection [T, H*d] or q, k, v side by side [T, 3*H*d].
 */
#define KDA_CONV_MAX_WIDTH 4

typedef enum { KDA_ACT_NONE = 0, KDA_ACT_SILU = 1 } kda_activation;

typedef struct {
    int32_t n_seqs;            /* N >= 0                                                 */
    int64_t total_tokens;      /* T = sum of the sequence lengths, < 2^31                */
    int32_t channels;          /* C, a multiple of 8                                     */
    int32_t width;             /* W, 1..KDA_CONV_MAX_WIDTH                               */
    int32_t activation;        /* kda_activation                                         */
    int32_t io_dtype;          /* kda_dtype of x, y and the states                       */
    const int32_t *cu_seqlens; /* [N+1] device offsets, or NULL = N equal sequences      */
    const void *x;             /* [T, C]                                                 */
    const float *weight;       /* [C, W]; weight[c, W-1] multiplies the current token    */
    const float *bias;         /* [C] or NULL (zero)                                     */
    const void *state_in;      /* [N, W-1, C] or NULL (zeros)                            */
    void *y;                   /* out [T, C]                                             */
    void *state_out;           /* out [N, W-1, C] or NULL; must not overlap state_in     */
} kda_conv_args;

typedef struct {
    kda_conv_args fwd;         /* the forward's arguments (y and state_out unused)       */
    const void *dy;            /* [T, C] io dtype                                        */
    const float *d_state_out;  /* [N, W-1, C] fp32 gradient of state_out, or NULL (zero) */
    float *dx;                 /* out [T, C] fp32                                        */
    float *dweight;            /* out [C, W] fp32                                        */
    float *dbias;              /* out [C] fp32, or NULL (not computed)                   */
    float *d_state_in;         /* out [N, W-1, C] fp32, or NULL (not computed)           */
    void *workspace;           /* kda_conv_bwd_workspace_size() bytes (per-CTA partials) */
    size_t workspace_bytes;
} kda_conv_bwd_args;

/* Decode / draft verification: L token slots per sequence, the state in place, with the
 * same slot conventions as kda_step (state_indices into a pool of n_slots states; slots
 * before first_slot[i] are padding that neither reads nor writes anything; the state is
 * advanced through accept_len[i] slots: the last W - 1 inputs of the committed tokens). */
typedef struct {
    int32_t n_seqs, steps;     /* N >= 0, L in 1..8                                      */
    int32_t channels, width, activation, io_dtype;   /* as in kda_conv_args              */
    const void *x;             /* [N, L, C]                                              */
    const float *weight;       /* [C, W]                                                 */
    const float *bias;         /* [C] or NULL                                            */
    void *state;               /* [n_slots, W-1, C] io dtype, updated in place           */
    const int32_t *state_indices;   /* [N] slot of each sequence, or NULL = slot i; the
                                       slots of sequences that commit must be distinct  */
    int32_t n_slots;           /* slots in the pool (N when state_indices is NULL)       */
    const int32_t *accept_len; /* [N] slots to commit (clamped to 0..L), or NULL = L     */
    const int32_t *first_slot; /* [N] padding slots before the tokens, or NULL = 0       */
    void *y;                   /* out [N, L, C]; padding slots are not written           */
    int32_t *dev_status;       /* NULL, or a device int32: KDA_ERR_INVALID_ARG when a
                                  state index is outside 0..n_slots-1 (that sequence is
                                  skipped)                                               */
} kda_conv_step_args;

kda_status kda_conv_fwd(const kda_conv_args *args, cudaStream_t stream);
kda_status kda_conv_bwd(const kda_conv_bwd_args *args, cudaStream_t stream);
size_t kda_conv_bwd_workspace_size(const kda_conv_bwd_args *args);
kda_status kda_conv_step(const kda_conv_step_args *args, cudaStream_t stream);

/*
 * kda_fwd_no_alloc -- kda_fwd for callers that cannot allocate device memory.
 * (This entry point has no counterpart in the pages; it is a deployment aid.)
 *
 * Some callers cannot call cudaMalloc, or any allocator, when they run the
 * forward: for example a plugin or callback executing inside another engine
 * that owns all device memory and passes it only the inputs and outputs, or a
 * latency-critical path that cannot afford cudaMalloc's implicit device
 * synchronisation. This call takes the same arguments as kda_fwd, ignores
 * args->workspace and args->workspace_bytes, and uses instead one file-scope
 * device array of KDA_NO_ALLOC_SCRATCH_BYTES bytes; it calls no allocator.
 *  - A problem whose kda_fwd_workspace_size() exceeds KDA_NO_ALLOC_SCRATCH_BYTES
 *    is rejected with KDA_ERR_INVALID_ARG before anything is enqueued.
 *  - Every GPU on which the array is loaded keeps it until the process exits.
 *  - The first call on a device looks up the array's device address with that
 *    device current (cudaGetSymbolAddress) and caches it; make that first call
 *    before any stream capture. A failed lookup returns KDA_ERR_CUDA.
 *  - All calls share the one array: calls whose work overlaps on the GPU (other
 *    streams or host threads) race. The array keeps the last call's contents;
 *    the forward writes every scratch byte before reading it, so nothing needs
 *    clearing between calls. For the same reason args->skip_prep, which would
 *    read chunk records an earlier call left in the scratch, is rejected with
 *    KDA_ERR_UNSUPPORTED.
 *  - The cached address is valid for the device's current context only: do not
 *    use this entry point across cudaDeviceReset (or a release and re-creation
 *    of the primary context).
 *  - The scratch holds the chunk table and the chunk records: per (chunk, head)
 *    66,048 bytes for bf16 I/O and 131,584 bytes for fp32 I/O, counted over
 *    (total_tokens / 64 + n_seqs) chunks. So (total_tokens / 64 + n_seqs) x heads
 *    may be at most about 4,060 (bf16) or 2,040 (fp32): at 96 heads one sequence
 *    of up to about 2,600 (bf16) or 1,280 (fp32) tokens. kda_fwd_workspace_size()
 *    gives the exact figure.
 * Outputs (o, hT, saved) are bit-identical to kda_fwd's on the same inputs.
 */
#define KDA_NO_ALLOC_SCRATCH_BYTES (256u * 1024u * 1024u)
kda_status kda_fwd_no_alloc(const kda_fwd_args *args, cudaStream_t stream);

/* Per-kernel timing hook for benchmarks. When `events` is not NULL, every later
 * kda_fwd / kda_bwd / kda_step call records events[i] on its stream right after
 * enqueueing its i-th stage (i < n_events): kda_fwd has 3 (chunk table, chunk prep,
 * state scan), kda_bwd 3 (chunk table, reverse dS scan, chunk-local gradients; for
 * fp32 I/O the second stage also re-runs the chunk prep and the third is two
 * kernels), kda_step 1. Elapsed times
 * between consecutive events (and one the caller records before the call) give
 * each kernel's device time. The caller owns the events and the array, which
 * must stay valid until the hook is cleared with kda_set_profile_events(NULL, 0).
 * Process-wide, not thread-safe; meant for single-threaded benchmarking. */
void kda_set_profile_events(cudaEvent_t *events, int32_t n_events);

/* Message of the last error on the calling host thread ("" if none). */
const char *kda_last_error(void);

/* Library ABI version (bumped on any change of the structs above). */
int32_t kda_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H */
