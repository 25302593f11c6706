// extern "C" entry points of libmtphead.so (declared and documented in include/mtp_head.h).
// Every argument is checked on the host before anything touches the GPU; a call that returns
// an error has launched nothing.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/mtp_head.h"
#include "common.cuh"
#include "internal.h"

namespace {

using mtp::kMaxB;
constexpr int kMaxContextRows = 65536;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int B, int H, int V) {
  if (B < 1 || B > kMaxB) return MTP_ERR_SHAPE;
  if (H < 1 || H > 65536) return MTP_ERR_SHAPE;
  if (V < 1) return MTP_ERR_SHAPE;
  return MTP_OK;
}

int check_eps(float eps) { return (eps >= 0.0f && !isinf(eps)) ? MTP_OK : MTP_ERR_ARG; }

int map_cuda(cudaError_t e) {
  if (e == cudaSuccess) return MTP_OK;
  if (e == cudaErrorNotSupported) return MTP_ERR_NOT_IMPLEMENTED;
  return MTP_ERR_CUDA;
}

int validate_input(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
                   const uint16_t* eh_proj, const int32_t* tokens, const uint16_t* target_hidden,
                   const uint16_t* x_out, const int32_t* status, int B, int H, int V, float eps) {
  if (!embed || !enorm_w || !hnorm_w || !eh_proj || !tokens || !target_hidden || !x_out)
    return MTP_ERR_ARG;
  if (check_eps(eps) != MTP_OK) return MTP_ERR_ARG;
  if (check_shape(B, H, V) != MTP_OK) return MTP_ERR_SHAPE;
  if (!aligned(embed, 16) || !aligned(enorm_w, 16) || !aligned(hnorm_w, 16) ||
      !aligned(eh_proj, 16) || !aligned(target_hidden, 16) || !aligned(x_out, 16) ||
      !aligned(tokens, 4) || (status && !aligned(status, 4)))
    return MTP_ERR_ALIGN;
  return MTP_OK;
}

int validate_output(const uint16_t* x, const uint16_t* final_norm_w, const void* lm_head,
                    const float* row_scale, int w_dtype, const float* logits, const int32_t* draft,
                    const int32_t* status, const void* workspace, size_t workspace_bytes, int B,
                    int H, int V, float eps) {
  if (!x || !final_norm_w || !lm_head || !draft) return MTP_ERR_ARG;
  if (w_dtype != MTP_W_BF16 && w_dtype != MTP_W_FP8_E4M3) return MTP_ERR_ARG;
  if (w_dtype == MTP_W_FP8_E4M3 && !row_scale) return MTP_ERR_ARG;
  if (check_eps(eps) != MTP_OK) return MTP_ERR_ARG;
  if (check_shape(B, H, V) != MTP_OK) return MTP_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(final_norm_w, 16) || !aligned(lm_head, 16) ||
      (row_scale && !aligned(row_scale, 4)) || (logits && !aligned(logits, 4)) ||
      !aligned(draft, 4) || (status && !aligned(status, 4)) || (workspace && !aligned(workspace, 16)))
    return MTP_ERR_ALIGN;
  if (!workspace || workspace_bytes < mtp::sweep_workspace_bytes(B)) return MTP_ERR_WORKSPACE;
  return MTP_OK;
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// Workspace of the whole-step entry points: the output stage's part, then room for the prebuilt
// concat of the batched input stage ([B, 2H] BF16, then [B] int32 row flags).
size_t step_concat_offset(int B) { return round256(mtp::sweep_workspace_bytes(B)); }
size_t step_workspace_bytes(int B, int H) {
  return step_concat_offset(B) + round256(static_cast<size_t>(B) * 2 * H * 2) + round256(static_cast<size_t>(B) * 4);
}

// cat_ws (may be null): workspace for a prebuilt concat, [B, 2H] BF16 then the [B] row flags
// 256-byte aligned after it.
int run_input(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
              const uint16_t* eh_proj, const int32_t* tokens, const uint16_t* target_hidden,
              uint16_t* x_out, int32_t* status, int B, int H, int V, float eps, void* stream,
              void* cat_ws = nullptr) {
  mtp::InputArgs a{};
  if (cat_ws != nullptr) {
    a.concat_ws = static_cast<uint16_t*>(cat_ws);
    a.valid_ws = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(cat_ws) + round256(static_cast<size_t>(B) * 2 * H * 2));
  }
  a.embed = embed;
  a.enorm_w = enorm_w;
  a.hnorm_w = hnorm_w;
  a.eh_proj = eh_proj;
  a.tokens = tokens;
  a.hidden = target_hidden;
  a.x = x_out;
  a.status = status;
  a.B = B;
  a.H = H;
  a.V = V;
  a.eps = eps;
  a.inv_h = 1.0 / static_cast<double>(H);
  return map_cuda(mtp::launch_input_stage(a, static_cast<cudaStream_t>(stream)));
}

int run_output(const uint16_t* x, const uint16_t* final_norm_w, const void* lm_head,
               const float* row_scale, int w_dtype, float* logits, int32_t* draft, int32_t* status,
               void* workspace, int B, int H, int V, float eps, void* stream) {
  mtp::SweepArgs a{};
  a.x = x;
  a.final_norm_w = final_norm_w;
  a.W = static_cast<const uint8_t*>(lm_head);
  a.scale = (w_dtype == MTP_W_FP8_E4M3) ? row_scale : nullptr;
  a.logits = logits;
  a.draft = draft;
  a.status = status;
  a.ws = static_cast<uint8_t*>(workspace);
  a.w_dtype = w_dtype;
  a.B = B;
  a.H = H;
  a.V = V;
  a.eps = eps;
  a.inv_h = 1.0 / static_cast<double>(H);
  return map_cuda(mtp::launch_sweep(a, static_cast<cudaStream_t>(stream)));
}

}  // namespace

namespace mtp {
// The output stage's host-side argument check, for other entry points of this library.
int check_output_args(const uint16_t* x, const uint16_t* final_norm_w, const void* lm_head,
                      const float* row_scale, int w_dtype, const float* logits, const int32_t* draft,
                      const int32_t* status, const void* workspace, size_t workspace_bytes, int B,
                      int H, int V, float eps) {
  return validate_output(x, final_norm_w, lm_head, row_scale, w_dtype, logits, draft, status,
                         workspace, workspace_bytes, B, H, V, eps);
}
}  // namespace mtp

extern "C" {

int mtp_head_input_batched(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
                           const uint16_t* eh_proj, const int32_t* tokens,
                           const uint16_t* target_hidden, uint16_t* x_out, int32_t* status, int B,
                           int H, int V, float eps, void* stream) {
  const int v = validate_input(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x_out,
                               status, B, H, V, eps);
  if (v != MTP_OK) return v;
  return run_input(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x_out, status, B, H, V,
                   eps, stream);
}

int mtp_head_input(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
                   const uint16_t* eh_proj, const int32_t* token, const uint16_t* target_hidden,
                   uint16_t* x_out, int32_t* status, int H, int V, float eps, void* stream) {
  return mtp_head_input_batched(embed, enorm_w, hnorm_w, eh_proj, token, target_hidden, x_out,
                                status, 1, H, V, eps, stream);
}

int mtp_head_logits_argmax_batched(const uint16_t* x, const uint16_t* final_norm_w,
                                   const void* lm_head, const float* row_scale, int w_dtype,
                                   float* logits, int32_t* draft, int32_t* status, void* workspace,
                                   size_t workspace_bytes, int B, int H, int V, float eps,
                                   void* stream) {
  const int v = validate_output(x, final_norm_w, lm_head, row_scale, w_dtype, logits, draft, status,
                                workspace, workspace_bytes, B, H, V, eps);
  if (v != MTP_OK) return v;
  return run_output(x, final_norm_w, lm_head, row_scale, w_dtype, logits, draft, status, workspace,
                    B, H, V, eps, stream);
}

int mtp_head_logits_argmax(const uint16_t* x, const uint16_t* final_norm_w, const void* lm_head,
                           const float* row_scale, int w_dtype, float* logits, int32_t* draft,
                           int32_t* status, void* workspace, size_t workspace_bytes, int H, int V,
                           float eps, void* stream) {
  return mtp_head_logits_argmax_batched(x, final_norm_w, lm_head, row_scale, w_dtype, logits, draft,
                                        status, workspace, workspace_bytes, 1, H, V, eps, stream);
}

size_t mtp_head_workspace_bytes(int B, int H, int V) {
  if (check_shape(B, H, V) != MTP_OK) return 0;
  return step_workspace_bytes(B, H);
}

int mtp_head_forward_batched(const uint16_t* embed, const uint16_t* enorm_w,
                             const uint16_t* hnorm_w, const uint16_t* eh_proj,
                             const uint16_t* final_norm_w, const void* lm_head,
                             const float* row_scale, int w_dtype, const int32_t* tokens,
                             const uint16_t* target_hidden, uint16_t* x, float* logits,
                             int32_t* draft, int32_t* status, void* workspace,
                             size_t workspace_bytes, int B, int H, int V, float eps, void* stream) {
  int v = validate_input(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x, status, B, H,
                         V, eps);
  if (v != MTP_OK) return v;
  v = validate_output(x, final_norm_w, lm_head, row_scale, w_dtype, logits, draft, status, workspace,
                      workspace_bytes, B, H, V, eps);
  if (v != MTP_OK) return v;
  // a workspace of the full size also takes the prebuilt concat of the batched input stage
  void* cat = workspace_bytes >= step_workspace_bytes(B, H) ? static_cast<uint8_t*>(workspace) + step_concat_offset(B)
                                                             : nullptr;
  v = run_input(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x, status, B, H, V, eps,
                stream, cat);
  if (v != MTP_OK) return v;
  return run_output(x, final_norm_w, lm_head, row_scale, w_dtype, logits, draft, status, workspace,
                    B, H, V, eps, stream);
}

int mtp_head_forward_host(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
                          const uint16_t* eh_proj, const uint16_t* final_norm_w,
                          const void* lm_head, const float* row_scale, int w_dtype,
                          const int32_t* tokens_host, const uint16_t* hidden_host,
                          int32_t* tokens_dev, uint16_t* hidden_dev, uint16_t* x_dev,
                          int32_t* draft_dev, int32_t* draft_host, int32_t* status,
                          void* workspace, size_t workspace_bytes, int B, int H, int V, float eps,
                          void* stream) {
  if (!tokens_host || !hidden_host || !draft_host) return MTP_ERR_ARG;
  int v = validate_input(embed, enorm_w, hnorm_w, eh_proj, tokens_dev, hidden_dev, x_dev, status, B,
                         H, V, eps);
  if (v != MTP_OK) return v;
  v = validate_output(x_dev, final_norm_w, lm_head, row_scale, w_dtype, nullptr, draft_dev, status,
                      workspace, workspace_bytes, B, H, V, eps);
  if (v != MTP_OK) return v;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(tokens_dev, tokens_host, sizeof(int32_t) * B, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MTP_ERR_CUDA;
  if (cudaMemcpyAsync(hidden_dev, hidden_host, sizeof(uint16_t) * static_cast<size_t>(B) * H,
                      cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MTP_ERR_CUDA;
  void* cat = workspace_bytes >= step_workspace_bytes(B, H) ? static_cast<uint8_t*>(workspace) + step_concat_offset(B)
                                                             : nullptr;
  v = run_input(embed, enorm_w, hnorm_w, eh_proj, tokens_dev, hidden_dev, x_dev, status, B, H, V,
                eps, stream, cat);
  if (v != MTP_OK) return v;
  v = run_output(x_dev, final_norm_w, lm_head, row_scale, w_dtype, nullptr, draft_dev, status,
                 workspace, B, H, V, eps, stream);
  if (v != MTP_OK) return v;
  if (cudaMemcpyAsync(draft_host, draft_dev, sizeof(int32_t) * B, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MTP_ERR_CUDA;
  int32_t dev_status = 0;
  if (status && cudaMemcpyAsync(&dev_status, status, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MTP_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MTP_ERR_CUDA;
  return dev_status;
}

size_t mtp_head_context_workspace_bytes(int R, int H) {
  if (R < 1 || R > kMaxContextRows || H < 1 || H > 65536) return 0;
  return mtp::context_workspace_bytes(R, H);
}

int mtp_head_context_rows(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
                          const uint16_t* eh_proj, const int32_t* tokens, const uint16_t* target_hidden,
                          uint16_t* x_out, int32_t* status, void* workspace, size_t workspace_bytes, int R,
                          int H, int V, float eps, void* stream) {
  if (!embed || !enorm_w || !hnorm_w || !eh_proj || !tokens || !target_hidden || !x_out) return MTP_ERR_ARG;
  if (check_eps(eps) != MTP_OK) return MTP_ERR_ARG;
  if (R < 1 || R > kMaxContextRows || H < 1 || H > 65536 || V < 1) return MTP_ERR_SHAPE;
  if (!aligned(embed, 16) || !aligned(enorm_w, 16) || !aligned(hnorm_w, 16) || !aligned(eh_proj, 16) ||
      !aligned(target_hidden, 16) || !aligned(x_out, 16) || !aligned(tokens, 4) ||
      (status && !aligned(status, 4)) || (workspace && !aligned(workspace, 16)))
    return MTP_ERR_ALIGN;
  if (R <= kMaxB) {  // a few rows: the batched input stage, one weight pass for all of them
    // its concat and row flags sit where this entry point's own kernels put them
    void* cat = (workspace && workspace_bytes >= mtp::context_workspace_bytes(R, H)) ? workspace : nullptr;
    return run_input(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x_out, status, R, H, V, eps,
                     stream, cat);
  }
  if (H % 32 != 0) return MTP_ERR_NOT_IMPLEMENTED;
  if (!workspace || workspace_bytes < mtp::context_workspace_bytes(R, H)) return MTP_ERR_WORKSPACE;
  mtp::ContextArgs a{};
  a.embed = embed;
  a.enorm_w = enorm_w;
  a.hnorm_w = hnorm_w;
  a.eh_proj = eh_proj;
  a.tokens = tokens;
  a.hidden = target_hidden;
  a.x = x_out;
  a.status = status;
  a.R = R;
  a.H = H;
  mtp::bind_context_workspace(&a, workspace);
  a.V = V;
  a.eps = eps;
  a.inv_h = 1.0 / static_cast<double>(H);
  return map_cuda(mtp::launch_context_rows(a, static_cast<cudaStream_t>(stream)));
}

int mtp_head_quantize_fp8(const uint16_t* w, uint8_t* q, float* row_scale, int32_t* status, int V,
                          int H, void* stream) {
  if (!w || !q || !row_scale || !status) return MTP_ERR_ARG;
  if (check_shape(1, H, V) != MTP_OK) return MTP_ERR_SHAPE;
  if (!aligned(w, 16) || !aligned(q, 16) || !aligned(row_scale, 4) || !aligned(status, 4))
    return MTP_ERR_ALIGN;
  return map_cuda(mtp::launch_quantize(w, q, row_scale, status, V, H, static_cast<cudaStream_t>(stream)));
}

const char* mtp_head_strerror(int status) {
  switch (status) {
    case MTP_OK: return "ok";
    case MTP_ERR_ARG: return "invalid argument (null pointer, unknown weight dtype, or eps not finite and >= 0)";
    case MTP_ERR_SHAPE: return "shape out of range (need 1 <= B <= 16, 1 <= H <= 65536, V >= 1)";
    case MTP_ERR_ALIGN: return "misaligned pointer (matrices and vectors need 16 bytes, int32/float 4 bytes)";
    case MTP_ERR_WORKSPACE: return "workspace missing or smaller than mtp_head_workspace_bytes()";
    case MTP_ERR_CUDA: return "CUDA runtime error while launching";
    case MTP_ERR_NONFINITE: return "the quantiser met a NaN or Inf weight; the FP8 copy is unusable";
    case MTP_ERR_TOKEN_RANGE: return "a token was outside [0, V); its x row was written as zeros";
    case MTP_ERR_NOT_IMPLEMENTED: return "no kernel for this shape combination in this build";
    case MTP_ERR_TIMEOUT: return "a kernel-side wait ran out of time";
    default: return "unknown status";
  }
}

}  // extern "C"
