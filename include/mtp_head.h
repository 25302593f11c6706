/*
 * mtp_head.h -- C ABI of libmtphead.so, the GB300 (sm_103a) hot path of the GLM-5.3 MTP
 * speculative draft head (the `Glm5NextMtpHead::forward_one` draft step).
 *
 * What it computes, for each of B independent sequences b (the decoder layer between the two
 * stages is the identity here; the source pages: "metrale_model_arch / glm5next_mtp_head.rs",
 * module doc math summary and `forward_one`):
 *
 *   input stage   c_b    = [ enorm(embed[token_b, :]) | hnorm(target_hidden_b) ]   [2H] BF16
 *                 x_b    = bf16( eh_proj . c_b )                                     [H]  BF16
 *   output stage  xhat_b = shared_head.norm(x_b)                                     [H]  BF16
 *                 logit_b[v] = lm_head[v, :] . xhat_b   (BF16 head, or the FP8 E4M3 copy
 *                              with per-row scale: s[v] * sum_k e4m3(Q[v, k]) * xhat_b[k])
 *                 draft_b = lowest v with logit_b[v] == max_u logit_b[u]
 *
 *   norm(x; w) = rms_norm_vanilla = bf16( x * w / sqrt(mean(x^2) + eps) )  -- never 1 + w
 *   ("metrale_model_arch / glm5next_layer / mod.rs", module doc invariant).
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless the argument says "host". The caller owns every
 *     buffer (weights, activations, outputs, workspace). The library allocates nothing and
 *     keeps no state beyond cached device attributes, with two stated exceptions: the pinned
 *     staging buffers and recorded graphs of mtp_head_forward_host, and the fixed workspace
 *     array of mtp_head_logits_argmax_batched_noalloc.
 *   - BF16 values are passed as uint16_t bit patterns, FP8 E4M3 codes as uint8_t (OCP E4M3
 *     "fn": bias 7, subnormals, max 448, no infinities). All matrices are row-major and dense.
 *   - Base pointers of matrices and vectors must be 16-byte aligned (every cudaMalloc /
 *     PyTorch allocation is); int32/float pointers 4-byte aligned. Misalignment returns
 *     MTP_ERR_ALIGN before anything is launched.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream) and the
 *     call returns without waiting, except mtp_head_forward_host, which is synchronous.
 *   - The return value reports host-checkable errors (arguments, shapes, alignment,
 *     workspace size) and launch failures (MTP_ERR_CUDA). Nothing is launched when it is not
 *     MTP_OK. Data-dependent errors (a token outside [0, V), a NaN/Inf weight handed to the
 *     quantiser, a kernel-side wait that gave up) are written by the kernels to the optional
 *     device word `status`: the first error stored wins; the caller zeroes it and reads it
 *     after synchronising. The library never clears it.
 *   - Shapes: 1 <= B <= 16, 1 <= H <= 65536, 1 <= V < 2^31, eps finite and >= 0.
 *   - Programmatic dependent launch: the input stage and the output stage are launched so that
 *     they may start streaming their weight matrix (eh_proj / lm_head) before the previous
 *     kernel on the stream has finished. They read tokens, target_hidden, x, the norm weights
 *     and the workspace only after it has finished. Do not write those two weight matrices in
 *     a kernel that itself triggers early launch of its dependents.
 */
#ifndef MTP_HEAD_H
#define MTP_HEAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MTP_OK = 0,
    MTP_ERR_ARG = -1,             /* null pointer, bad enum, eps not finite or negative */
    MTP_ERR_SHAPE = -2,           /* B, H or V outside the supported range */
    MTP_ERR_ALIGN = -3,           /* a pointer is not aligned as stated above */
    MTP_ERR_WORKSPACE = -4,       /* workspace NULL or smaller than mtp_head_workspace_bytes */
    MTP_ERR_CUDA = -5,            /* a CUDA runtime call or launch failed */
    MTP_ERR_NONFINITE = -6,       /* (device status) the quantiser met a NaN or Inf weight */
    MTP_ERR_TOKEN_RANGE = -7,     /* (device status) a token outside [0, V) */
    MTP_ERR_NOT_IMPLEMENTED = -8, /* shape combination without a kernel in this build */
    MTP_ERR_TIMEOUT = -9          /* (device status) a kernel-side wait ran out of time */
} mtp_status;

enum { MTP_W_BF16 = 0, MTP_W_FP8_E4M3 = 1 };

/* ------------------------------------------------------------------------------------------
 * Input stage ("glm5next_mtp_head.rs", `forward_one`: the embedding row read by pointer at
 * token*hidden, `norm` with enorm into concat[0:H] and hnorm into concat[H:2H], then the
 * `eh_proj` dense gemv with n = H, k = 2H). One fused kernel per call.
 *
 *   embed          [V, H]  BF16   token embedding table (row token_b is gathered)
 *   enorm_w        [H]     BF16   enorm weight
 *   hnorm_w        [H]     BF16   hnorm weight
 *   eh_proj        [H, 2H] BF16   projection; row n is output n, columns [0:H) meet the enorm
 *                                 half of the concat, [H:2H) the hnorm half
 *   tokens         [B]     int32  device-resident tokens (a graph replay or a draft chain
 *                                 can feed the previous draft straight back in)
 *   target_hidden  [B, H]  BF16   the target model's hidden state for each sequence
 *   x_out          [B, H]  BF16   output: the block input x
 *   status         [1]     int32  optional (may be NULL); MTP_ERR_TOKEN_RANGE if some token is
 *                                 outside [0, V): that sequence's x row is written as zeros and
 *                                 the embedding table is not read for it
 * ---------------------------------------------------------------------------------------- */
int mtp_head_input_batched(const uint16_t* embed, const uint16_t* enorm_w,
                           const uint16_t* hnorm_w, const uint16_t* eh_proj,
                           const int32_t* tokens, const uint16_t* target_hidden,
                           uint16_t* x_out, int32_t* status, int B, int H, int V, float eps,
                           void* stream);

/* Same, B = 1. */
int mtp_head_input(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
                   const uint16_t* eh_proj, const int32_t* token, const uint16_t* target_hidden,
                   uint16_t* x_out, int32_t* status, int H, int V, float eps, void* stream);

/* ------------------------------------------------------------------------------------------
 * Context-row input stage ("glm5next_mtp_head.rs", `rows_impl`: for every context row r, the
 * embedding row of tokens[r] and target_hidden row r go through enorm / hnorm, the concat and
 * eh_proj -- the input stage of `forward_one` per row; the source loops over the rows on the
 * host, here all R rows run at once).
 *
 *   embed, enorm_w, hnorm_w, eh_proj  as for mtp_head_input_batched
 *   tokens         [R]     int32  device-resident tokens; tokens[r] is the token row r pairs
 *                                 with (the source pairs hidden row r with the token after it,
 *                                 so a caller passes its token array shifted by one)
 *   target_hidden  [R, H]  BF16
 *   x_out          [R, H]  BF16   output; a row whose token is outside [0, V) is zeros and
 *                                 status (optional) gets MTP_ERR_TOKEN_RANGE
 *   workspace             device scratch of at least mtp_head_context_workspace_bytes(R, H)
 *                         bytes (no initialisation needed; may be NULL when R <= 16, in which
 *                         case the batched input stage normalises the rows in every CTA)
 *   R              1 .. 65536 rows
 *
 * With the workspace (and H a multiple of 32, R >= 2) two kernels run: the normalised concat of
 * every row into the workspace (the same correctly rounded BF16 values as the input stage), then
 * x = concat . eh_proj^T as a tiled GEMM on the tcgen05 tensor cores with FP32 accumulation --
 * the source's eh_proj precision, so x is the BF16 rounding of an FP32-accumulated sum -- plus,
 * when the GEMM splits its tiles along k, a kernel that adds their partial sums in k order.
 * R <= 16 without the workspace (or with H not a multiple of 32, or R = 1) runs the input stage
 * of mtp_head_input_batched instead. H must be a multiple of 32 for R > 16
 * (MTP_ERR_NOT_IMPLEMENTED otherwise).
 * ---------------------------------------------------------------------------------------- */
int mtp_head_context_rows(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
                          const uint16_t* eh_proj, const int32_t* tokens, const uint16_t* target_hidden,
                          uint16_t* x_out, int32_t* status, void* workspace, size_t workspace_bytes,
                          int R, int H, int V, float eps, void* stream);

/* Bytes of workspace mtp_head_context_rows needs for R rows (0 for invalid shapes). */
size_t mtp_head_context_workspace_bytes(int R, int H);

/* ------------------------------------------------------------------------------------------
 * Output stage ("glm5next_mtp_head.rs", `forward_one`: `shared_head.norm` in place, then the
 * `lm_head` dense gemv -- or `dense_gemv_fp8w` over the FP8 copy described in the `head_fp8`
 * doc -- then `argmax_bf16`; here the sweep covers the whole vocabulary on one GPU and the
 * argmax is fused into it). One sweep kernel per call, which reads lm_head once for all B
 * sequences; for B = 2..16 a small kernel before it sums the squares of x's rows (for the norm).
 *
 *   x              [B, H]  BF16   block output
 *   final_norm_w   [H]     BF16   shared_head.norm weight
 *   lm_head        [V, H]  BF16 (w_dtype MTP_W_BF16) or E4M3 codes (MTP_W_FP8_E4M3)
 *   row_scale      [V]     fp32   per-row scale of the FP8 copy; NULL for BF16
 *   logits         [B, V]  fp32   optional output (NULL = not stored). Kept in fp32, not BF16.
 *   draft          [B]     int32  output: lowest index of the maximum logit; NaN never wins;
 *                                 -1 if every logit of that sequence is NaN
 *   status         [1]     int32  optional (may be NULL); MTP_ERR_TIMEOUT on a kernel-side wait
 *   workspace             device scratch of at least mtp_head_workspace_bytes(B, H, V)
 *                         bytes, zero-filled once before its first use. The kernels return
 *                         its counters to zero themselves, so it stays valid across calls and
 *                         CUDA-graph replays. Two calls that may run at the same time
 *                         (different streams) need different workspaces.
 * ---------------------------------------------------------------------------------------- */
int mtp_head_logits_argmax_batched(const uint16_t* x, const uint16_t* final_norm_w,
                                   const void* lm_head, const float* row_scale, int w_dtype,
                                   float* logits, int32_t* draft, int32_t* status,
                                   void* workspace, size_t workspace_bytes, int B, int H, int V,
                                   float eps, void* stream);

/* Same, B = 1. */
int mtp_head_logits_argmax(const uint16_t* x, const uint16_t* final_norm_w, const void* lm_head,
                           const float* row_scale, int w_dtype, float* logits, int32_t* draft,
                           int32_t* status, void* workspace, size_t workspace_bytes, int H,
                           int V, float eps, void* stream);

/* ------------------------------------------------------------------------------------------
 * Output stage over one vocabulary shard ("glm5next_mtp_head.rs": the vocab-shard geometry
 * `head_rank` / `head_v0` / `head_n` -- a rank sweeps rows [head_v0, head_v0 + head_n) of the
 * shared lm_head, and its FP8 copy covers that shard only -- and `forward_one`'s sharded branch
 * with its cross-rank pick). The same kernels as mtp_head_logits_argmax_batched, over the n rows
 * that start at global row v0:
 *
 *   lm_head_shard    [n, H]  BF16 or E4M3 codes: the shard's rows (row v0 of the full matrix;
 *                            16-byte aligned, as for the output stage)
 *   row_scale_shard  [n]     fp32 scales of those rows (FP8), NULL for BF16
 *   v0, n                    the shard's first global row and its row count; 0 <= v0,
 *                            1 <= n, v0 + n <= 2^31 - 1 (else MTP_ERR_SHAPE)
 *   logits           [B, n]  fp32, optional: the shard's logits (column j is global row v0 + j)
 *   pick             [B]     int64 output, 8-byte aligned: each sequence's exchange key of its
 *                            (max logit, lowest global index) over the shard -- see below
 *   draft            [B]     int32, optional: the shard's own draft as a global index
 *   x, final_norm_w, status, workspace, B, H, eps, stream   as for the output stage
 *
 * Exchange key. One int64 per sequence whose signed order is the argmax order: the larger FP32
 * value first, then the lower global index (-0 counts as +0). The pick over any set of shards is
 * therefore the plain maximum of their keys -- mtp_head_pick_combine on one GPU, or a MAX
 * all-reduce of the [B] keys between ranks -- exact and for any number of shards. The source
 * exchanges BF16 lanes (each rank's max logit and three base-256 digits of its index) through a
 * SUM all-reduce, because its all-reduce sums BF16 elements; with FP32 logits a BF16 lane would
 * round two close maxima to one value, so the key carries the FP32 value whole. A shard whose
 * logits are all NaN gives the empty key INT64_MIN, below every other key.
 * ---------------------------------------------------------------------------------------- */
int mtp_head_logits_argmax_shard(const uint16_t* x, const uint16_t* final_norm_w,
                                 const void* lm_head_shard, const float* row_scale_shard,
                                 int w_dtype, int v0, int n, float* logits, int64_t* pick,
                                 int32_t* draft, int32_t* status, void* workspace,
                                 size_t workspace_bytes, int B, int H, float eps, void* stream);

/* The pick over R shards: picks [R, B] int64 (row r = shard r's keys, 8-byte aligned) ->
 * draft [B] int32 (the global index of the largest key; -1 when every key of that sequence is
 * empty) and value [B] fp32 (optional, may be NULL: the winning logit). One small kernel on
 * `stream`; 1 <= R <= 65536, 1 <= B <= 16. After a MAX all-reduce between ranks, R = 1 decodes. */
int mtp_head_pick_combine(const int64_t* picks, int R, int B, int32_t* draft, float* value,
                          void* stream);

/* The exchange key on the host (no GPU involved): the key of (value, global index), and its
 * index and value back. mtp_head_pick_key returns INT64_MIN for index < 0 or a NaN value;
 * mtp_head_pick_index returns -1 and mtp_head_pick_value NaN for that key. */
int64_t mtp_head_pick_key(float value, int32_t index);
int32_t mtp_head_pick_index(int64_t key);
float mtp_head_pick_value(int64_t key);

/* ------------------------------------------------------------------------------------------
 * Output stage without a caller-provided workspace. The source pages have no counterpart: this
 * entry point exists for callers of this library that cannot allocate device memory -- e.g. a
 * plug-in that only receives the buffers its host framework hands it and has no allocator of
 * its own, or a process whose device memory was all claimed up front by another allocator.
 * It computes exactly what mtp_head_logits_argmax_batched computes (same kernels, same
 * arguments minus workspace / workspace_bytes) and allocates nothing: the workspace is a fixed
 * device array inside the library, 2,304 bytes, enough for any batch (B <= 16);
 * every GPU that loads the library holds it until the process exits. B outside 1..16 returns
 * MTP_ERR_SHAPE before anything runs.
 *   - The first call on a device looks up that array's device address (once per device, with
 *     the device current). Make that first call before any stream capture on the device. The
 *     address is kept for the life of the process: after cudaDeviceReset (or any reset of the
 *     device's primary context) the library's device array is a new one and the kept address is
 *     stale, so do not call this entry point on a device after resetting it.
 *   - All calls share the one array. The call clears its counter on `stream` before launching,
 *     so it never depends on what a previous call left there, but calls that may run at the
 *     same time on the GPU (different streams, or different host threads) race on it: order
 *     them on one stream or use mtp_head_logits_argmax_batched with separate workspaces. The
 *     clearing is a memset between the preceding kernel and the sweep, so unlike the workspace
 *     entry point the sweep cannot start its weight stream before the preceding kernel ends.
 * ---------------------------------------------------------------------------------------- */
int mtp_head_logits_argmax_batched_noalloc(const uint16_t* x, const uint16_t* final_norm_w,
                                           const void* lm_head, const float* row_scale,
                                           int w_dtype, float* logits, int32_t* draft,
                                           int32_t* status, int B, int H, int V, float eps,
                                           void* stream);

/* Bytes of workspace for the output stage and the whole-step entry points (no device query; 0
 * for invalid shapes): the output stage's part (the first 2304 bytes for any B, which must be
 * zero-filled once), then, 256-byte aligned, room for the context-row path's workspace of B rows
 * (mtp_head_context_workspace_bytes(B, H): concat, row flags and FP32 partial sums; no
 * initialisation needed). The output stage alone accepts any workspace of at least its own part.
 * mtp_head_forward_batched / _host given a workspace of the full size run the input stage of
 * 2..16 sequences at H a multiple of 32 through the context-row path (mtp_head_context_rows:
 * concat kernel + tcgen05 GEMM; x then carries the GEMM's FP32 accumulation); otherwise they run
 * the input stage of mtp_head_input_batched. */
size_t mtp_head_workspace_bytes(int B, int H, int V);

/* ------------------------------------------------------------------------------------------
 * Whole draft step, device buffers: the input stage into x, then the output stage from x.
 * Exactly mtp_head_input_batched followed by mtp_head_logits_argmax_batched on one stream.
 * ---------------------------------------------------------------------------------------- */
int mtp_head_forward_batched(const uint16_t* embed, const uint16_t* enorm_w,
                             const uint16_t* hnorm_w, const uint16_t* eh_proj,
                             const uint16_t* final_norm_w, const void* lm_head,
                             const float* row_scale, int w_dtype, const int32_t* tokens,
                             const uint16_t* target_hidden, uint16_t* x, float* logits,
                             int32_t* draft, int32_t* status, void* workspace,
                             size_t workspace_bytes, int B, int H, int V, float eps,
                             void* stream);

/* ------------------------------------------------------------------------------------------
 * Whole draft step from HOST buffers, synchronous: the shape of the source's
 * `forward_one(token, hidden_in, ...) -> u32`, which synchronises and copies the draft to the
 * host. Copies tokens_host [B] and hidden_host [B, H] into the caller's device buffers
 * tokens_dev / hidden_dev, runs mtp_head_forward_batched, copies draft back into
 * draft_host [B] and waits for the stream. Host buffers should be pinned for asynchronous
 * copies. The device `status` word, if given, is read back too and returned when nonzero.
 *
 * On a stream other than the legacy default stream (and not under the caller's own capture),
 * the first call for a given set of device buffers, shapes, eps and stream runs operation by
 * operation and then records the step in a CUDA graph around small mapped pinned staging
 * buffers (held by the library, at most 8 such steps, least recently used replaced). Later calls
 * with the same set copy the host inputs into the staging buffers, launch the graph once, wait,
 * and copy the draft out: the same work, without a launch per operation. Inside the graph the
 * moves between the staging buffers and tokens_dev / hidden_dev / draft_dev are small kernels
 * on the mapped memory (when B * H is a multiple of 8; copy operations otherwise). The host buffers may
 * differ from call to call. Calls from several threads are safe; calls sharing a recorded
 * step are serialised. On that recorded path the call returns as soon as the step's last kernel
 * has written the draft and status to the staging memory and set a completion word there (the
 * host polls it, asking the stream now and then so that a failed launch returns MTP_ERR_CUDA),
 * which spares the wake-up of a stream synchronisation; the stream may then still be retiring
 * that kernel, so work on another stream that must follow this step should wait on `stream`.
 * ---------------------------------------------------------------------------------------- */
int mtp_head_forward_host(const uint16_t* embed, const uint16_t* enorm_w,
                          const uint16_t* hnorm_w, const uint16_t* eh_proj,
                          const uint16_t* final_norm_w, const void* lm_head,
                          const float* row_scale, int w_dtype,
                          const int32_t* tokens_host, const uint16_t* hidden_host,
                          int32_t* tokens_dev, uint16_t* hidden_dev, uint16_t* x_dev,
                          int32_t* draft_dev, int32_t* draft_host, int32_t* status,
                          void* workspace, size_t workspace_bytes, int B, int H, int V,
                          float eps, void* stream);

/* ------------------------------------------------------------------------------------------
 * The same step with the arguments that stay fixed from call to call gathered in one struct
 * (no counterpart on the source pages, like mtp_head_forward_host itself, whose shape is
 * `forward_one`'s). For a caller that makes the same draft step over and over through a costly
 * call boundary -- a language binding marshals 23 arguments per call, ~3 us from Python --
 * a step then passes four. The fields mean what the parameters of mtp_head_forward_host of the
 * same names mean; mtp_head_forward_host_args(a, tokens_host, hidden_host, draft_host) is
 * exactly mtp_head_forward_host(a->embed, ..., tokens_host, hidden_host, a->tokens_dev, ...,
 * draft_host, a->status, ..., a->stream): the same work, results and status codes, plus
 * MTP_ERR_ARG for a NULL `a`. The struct is read during the call only.
 * ---------------------------------------------------------------------------------------- */
typedef struct mtp_host_step_args {
  const uint16_t* embed;
  const uint16_t* enorm_w;
  const uint16_t* hnorm_w;
  const uint16_t* eh_proj;
  const uint16_t* final_norm_w;
  const void* lm_head;
  const float* row_scale;
  int w_dtype;
  int32_t* tokens_dev;
  uint16_t* hidden_dev;
  uint16_t* x_dev;
  int32_t* draft_dev;
  int32_t* status;
  void* workspace;
  size_t workspace_bytes;
  int B;
  int H;
  int V;
  float eps;
  void* stream;
} mtp_host_step_args;

int mtp_head_forward_host_args(const mtp_host_step_args* a, const int32_t* tokens_host,
                               const uint16_t* hidden_host, int32_t* draft_host);

/* ------------------------------------------------------------------------------------------
 * FP8 E4M3 copy of a [V, H] BF16 matrix ("glm5next_mtp_head.rs", `head_fp8` doc: an E4M3
 * copy of lm_head used for drafting only). Per row v:
 *   row_scale[v] = fp32( max_k |w[v, k]| / 448 )
 *   q[v, k]      = e4m3_rne_satfinite( fp32( w[v, k] / row_scale[v] ) )
 * An all-zero row gives scale 0 and zero codes. A NaN or Inf weight stores
 * MTP_ERR_NONFINITE in `status` (required here) and that row's codes and scale as zeros; the
 * copy must then not be used (the source's "quantisation fails" case).
 *   w [V, H] BF16 -> q [V, H] uint8 (E4M3 codes), row_scale [V] fp32
 * ---------------------------------------------------------------------------------------- */
int mtp_head_quantize_fp8(const uint16_t* w, uint8_t* q, float* row_scale, int32_t* status,
                          int V, int H, void* stream);

/* ------------------------------------------------------------------------------------------
 * Give-up time of the kernels' stage waits (no counterpart on the source pages, which have no
 * device-side waits: this library's kernels wait on shared-memory barriers for their weight
 * copies and for each other's stages, and every such wait is bounded so that a stalled copy can
 * never hang the GPU). Past the limit the kernel stores MTP_ERR_TIMEOUT in `status`, lets its own
 * copies in flight land, and returns; the draft and logits of that call are then undefined, and
 * the workspace is left ready for the next call. Default 2 s (2000000000 ns), far above any
 * real wait. The limit applies to the output-stage kernels (every batch size) and to the
 * single-sequence input stage, launched after this call (a CUDA graph keeps the limit it was
 * recorded with); the batched input stage and the context-row kernels always use 2 s, and so
 * does every wait for a kernel's own copies before it exits. Process-wide; returns the previous
 * limit. A short limit (a few ns: the device clock it is compared with advances about once a
 * microsecond) makes the waits that find their data missing run out; ns = 0 makes every stage
 * wait give up at once, whatever the data. Both put the error path within reach of a test.
 * ---------------------------------------------------------------------------------------- */
unsigned long long mtp_head_set_wait_limit_ns(unsigned long long ns);

/* Static description of a status code (never NULL). */
const char* mtp_head_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* MTP_HEAD_H */
