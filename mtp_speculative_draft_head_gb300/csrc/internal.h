// Host-side declarations shared by the translation units of libmtphead.so.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched through the runtime)
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mtp {

// Tuning constants of the streaming kernels (compile-time; see the kernels for their use).
#ifndef MTP_WARPS
#define MTP_WARPS 8
#endif
#ifndef MTP_CHUNK
#define MTP_CHUNK 4096
#endif
#ifndef MTP_MAX_STAGES
#define MTP_MAX_STAGES 6
#endif
#ifndef MTP_MIXED_FMA
#define MTP_MIXED_FMA 1
#endif
#ifndef MTP_REGX
#define MTP_REGX 1
#endif
#ifndef MTP_TC_MIN_B
#define MTP_TC_MIN_B 2  // smallest batch the tensor-core output stage takes
#endif

constexpr int kWarps = MTP_WARPS;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = MTP_CHUNK;        // bytes per pipeline stage
constexpr int kMaxStages = MTP_MAX_STAGES;
constexpr int kTmaMaxB = 4;              // the CUDA-core streaming kernels take B <= 4

constexpr int kSmemReserve = 1024;      // opt-in bytes kept back for static shared variables
// shared scratch of the norm prologue: up to 2 * 16 vectors, (2 * warps + 2) floats each
constexpr size_t kRedBytes = sizeof(float) * 2 * 16 * (2 * kWarps + 2);

struct DeviceInfo {
  int sm_count;
  int smem_optin;  // dynamic shared memory a block may use (opt-in maximum - kSmemReserve)
};

// Cached per device; returns cudaSuccess or the error of the first query.
cudaError_t device_info(DeviceInfo* info);

// Give-up time of the stage waits of the kernels launched from now on (process-wide, 2 s by
// default); set_stage_wait_ns returns the previous value.
unsigned long long stage_wait_ns();
unsigned long long set_stage_wait_ns(unsigned long long ns);

// cudaLaunchKernelExC with programmatic stream serialization allowed; raises the kernel's
// dynamic shared memory limit once per device. device_info() must have been called first.
cudaError_t launch_pdl(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void** args);

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry point (so the
// library does not link against libcuda); nullptr if the driver does not provide it.
using TmapEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
TmapEncodeFn tensor_map_encoder();

struct InputArgs {
  const uint16_t* embed;
  const uint16_t* enorm_w;
  const uint16_t* hnorm_w;
  const uint16_t* eh_proj;
  const int32_t* tokens;
  const uint16_t* hidden;
  uint16_t* x;
  int32_t* status;
  int B, H, V;
  float eps;
  double inv_h;  // 1 / H (fp64), for the mean of squares
  int stages;  // pipeline stages (bulk-copy kernel)
  int group;   // sequences whose concat is resident at once (plain kernel)
  unsigned long long wait_ns;  // give-up time of the single-sequence kernel's stage waits
};

struct SweepArgs {
  const uint16_t* x;
  const uint16_t* final_norm_w;
  const uint8_t* W;      // lm_head bytes (BF16 pairs or E4M3 codes)
  const float* scale;    // FP8 row scales or nullptr
  float* logits;         // may be nullptr
  int32_t* draft;        // may be nullptr when pick is given
  int32_t* status;
  uint8_t* ws;
  int w_dtype;
  int B, H, V;
  float eps;
  double inv_h;  // 1 / H (fp64), for the mean of squares
  int stages;
  // Vocabulary shard: W (and scale) start at global row index_base, V is the shard's row count;
  // the draft is a global index, and pick (may be nullptr) receives each sequence's exchange key.
  int32_t index_base;
  int64_t* pick;
  unsigned long long wait_ns;  // give-up time of the stage waits
};

struct ContextArgs {
  const uint16_t* embed;
  const uint16_t* enorm_w;
  const uint16_t* hnorm_w;
  const uint16_t* eh_proj;
  const int32_t* tokens;
  const uint16_t* hidden;
  uint16_t* x;
  int32_t* status;
  uint16_t* concat;  // workspace: [R, 2H] BF16
  int32_t* valid;    // workspace: [R] token-in-range flags
  float* partial;    // workspace: FP32 partial sums of tiles shared between CTAs
  int R, H, V;
  float eps;
  double inv_h;
};

// Context rows (R >= 1, H a multiple of 32): concat kernel + tensor-core GEMM (+ the in-order sum
// of the partials of tiles whose k range was shared between CTAs).
cudaError_t launch_context_rows(const ContextArgs& a, cudaStream_t stream);
// The first kernel of that path alone: the normalised concat rows and row flags into
// a.concat / a.valid.
cudaError_t launch_context_concat(const ContextArgs& a, cudaStream_t stream);
// Workspace of the context-row stage: bytes needed, and pointing a's workspace fields into ws.
size_t context_workspace_bytes(int R, int H);
void bind_context_workspace(ContextArgs* a, void* ws);

cudaError_t launch_input_stage(const InputArgs& a, cudaStream_t stream);
// Batched (2 <= B <= 16) input stage on tensor cores; *launched stays false when the shape is
// not supported (H not a multiple of 8, not enough shared memory).
cudaError_t launch_input_tc(const InputArgs& a, cudaStream_t stream, bool* launched);
cudaError_t launch_sweep(const SweepArgs& a, cudaStream_t stream);
// Batched (2 <= B <= 16) output stage on tensor cores; *launched stays false when the shape is
// not supported (H not a multiple of 8, no tensor-map encoder, not enough shared memory).
cudaError_t launch_sweep_tc(const SweepArgs& a, cudaStream_t stream, bool* launched);
// The host-buffer step's moves as kernels on mapped pinned memory (device addresses of host
// buffers): hidden [B, H] (B * H a multiple of 8) and tokens in; draft and status (may be null) out,
// then the completion word seq_out set to *seq_in (both may be null).
cudaError_t launch_host_in(const int32_t* tok_src, const uint16_t* hid_src, int32_t* tok_dst, uint16_t* hid_dst,
                           int B, int H, cudaStream_t stream);
cudaError_t launch_host_out(const int32_t* draft_src, int32_t* draft_dst, const int32_t* status_src, int32_t* status_dst,
                            int B, const uint32_t* seq_in, uint32_t* seq_out, cudaStream_t stream);
cudaError_t launch_quantize(const uint16_t* w, uint8_t* q, float* scale, int32_t* status,
                            int V, int H, cudaStream_t stream);
// Pick over R shards' exchange keys picks[r * B + b]: draft[b] (global index, -1 if empty) and
// optionally value[b].
cudaError_t launch_pick_combine(const int64_t* picks, int R, int B, int32_t* draft, float* value,
                                cudaStream_t stream);

// Host-side argument check of the output stage (status code, nothing launched).
int check_output_args(const uint16_t* x, const uint16_t* final_norm_w, const void* lm_head,
                      const float* row_scale, int w_dtype, const float* logits, const int32_t* draft,
                      const int32_t* status, const void* workspace, size_t workspace_bytes, int B,
                      int H, int V, float eps);

// Bytes of the output stage's workspace, the same for every B (2304: the CTA completion counter,
// the row counter of the single-sequence sweep, each sequence's running pick, the batched
// sweep's norm parts).
size_t sweep_workspace_bytes(int B);

}  // namespace mtp
