// extern "C" entry points of libmtphead.so (declared and documented in include/mtp_head.h).
// Every argument is checked on the host before anything touches the GPU; a call that returns
// an error has launched nothing.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <memory>
#include <mutex>
#include <vector>

#include "../../include/mtp_head.h"
#include "common.cuh"
#include "internal.h"
#include "host_back.h"

namespace {

using mtp::kMaxB;
constexpr int kMaxContextRows = 65536;
constexpr int kMaxPickShards = 65536;  // picks combined by one mtp_head_pick_combine call

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
                    int H, int V, float eps, bool draft_optional = false) {
  if (!x || !final_norm_w || !lm_head || (!draft && !draft_optional)) return MTP_ERR_ARG;
  if (w_dtype != MTP_W_BF16 && w_dtype != MTP_W_FP8_E4M3) return MTP_ERR_ARG;
  if (w_dtype == MTP_W_FP8_E4M3 && !row_scale) return MTP_ERR_ARG;
  if (check_eps(eps) != MTP_OK) return MTP_ERR_ARG;
  if (check_shape(B, H, V) != MTP_OK) return MTP_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(final_norm_w, 16) || !aligned(lm_head, 16) ||
      (row_scale && !aligned(row_scale, 4)) || (logits && !aligned(logits, 4)) ||
      (draft && !aligned(draft, 4)) || (status && !aligned(status, 4)) || (workspace && !aligned(workspace, 16)))
    return MTP_ERR_ALIGN;
  if (!workspace || workspace_bytes < mtp::sweep_workspace_bytes(B)) return MTP_ERR_WORKSPACE;
  return MTP_OK;
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// Workspace of the whole-step entry points: the output stage's part, then room for the context-row
// path's workspace for B rows (concat, row flags, FP32 partials).
size_t step_concat_offset(int B) { return round256(mtp::sweep_workspace_bytes(B)); }
size_t step_workspace_bytes(int B, int H) { return step_concat_offset(B) + mtp::context_workspace_bytes(B, H); }

int run_input(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
              const uint16_t* eh_proj, const int32_t* tokens, const uint16_t* target_hidden,
              uint16_t* x_out, int32_t* status, int B, int H, int V, float eps, void* stream) {
  mtp::InputArgs a{};
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
  a.wait_ns = mtp::stage_wait_ns();
  return map_cuda(mtp::launch_input_stage(a, static_cast<cudaStream_t>(stream)));
}

// The context-row path into x_out: the normalised concat of every row into ws, then
// x = concat . eh_proj^T on the tcgen05 tensor cores (FP32 accumulation), plus the in-order sum of
// the partials of tiles split along k. H must be a multiple of 32; ws holds
// context_workspace_bytes(R, H).
int run_context(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
                const uint16_t* eh_proj, const int32_t* tokens, const uint16_t* target_hidden,
                uint16_t* x_out, int32_t* status, int R, int H, int V, float eps, void* stream, void* ws) {
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
  mtp::bind_context_workspace(&a, ws);
  a.V = V;
  a.eps = eps;
  a.inv_h = 1.0 / static_cast<double>(H);
  return map_cuda(mtp::launch_context_rows(a, static_cast<cudaStream_t>(stream)));
}

// Input stage of the whole-step entry points. With room for the context-row workspace after the
// output stage's part (a workspace of mtp_head_workspace_bytes), 2..16 sequences at H % 32 == 0 take
// the context-row path: its GEMM streams eh_proj from every SM and measured 26-27 us for B = 4..16
// at H = 6144, against 36-38 us for the mma.sync kernel, whose per-stage MMA work held each CTA to
// ~34 GB/s. ws_ctx may be null (no room): then the batched input stage runs.
int run_step_input(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
                   const uint16_t* eh_proj, const int32_t* tokens, const uint16_t* target_hidden,
                   uint16_t* x_out, int32_t* status, int B, int H, int V, float eps, void* stream, void* ws_ctx) {
  if (ws_ctx != nullptr && B >= 2 && H % 32 == 0)
    return run_context(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x_out, status, B, H, V, eps, stream,
                       ws_ctx);
  return run_input(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x_out, status, B, H, V, eps, stream);
}

// index_base / pick: a vocabulary shard's first global row and its exchange keys (may be null).
mtp::SweepArgs output_args(const uint16_t* x, const uint16_t* final_norm_w, const void* lm_head,
                           const float* row_scale, int w_dtype, float* logits, int32_t* draft, int32_t* status,
                           void* workspace, int B, int H, int V, float eps, int32_t index_base = 0,
                           int64_t* pick = nullptr) {
  mtp::SweepArgs a{};
  a.index_base = index_base;
  a.pick = pick;
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
  a.wait_ns = mtp::stage_wait_ns();
  return a;
}

int run_output(const uint16_t* x, const uint16_t* final_norm_w, const void* lm_head,
               const float* row_scale, int w_dtype, float* logits, int32_t* draft, int32_t* status,
               void* workspace, int B, int H, int V, float eps, void* stream, int32_t index_base = 0,
               int64_t* pick = nullptr) {
  const mtp::SweepArgs a = output_args(x, final_norm_w, lm_head, row_scale, w_dtype, logits, draft, status,
                                       workspace, B, H, V, eps, index_base, pick);
  return map_cuda(mtp::launch_sweep(a, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------------------------------
// The host-buffer whole step. Each call copies the inputs in, runs both stages, copies the draft
// out and waits, like the source's forward_one. Launching those five or six operations one by
// one costs several microseconds of host time each, and the GPU idles meanwhile, so the first
// call for a given set of device buffers, shapes and stream runs directly and then records the
// step in a CUDA graph around small pinned staging buffers; later calls copy the host inputs into
// the staging buffers (a few KB), launch the graph once, wait, and copy the draft out. A stream
// that is the legacy default stream, or is being captured by the caller, always runs directly.
struct HostStep {
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
  int B, H, V;
  float eps;
  cudaStream_t stream;

  bool same(const HostStep& o) const {
    return embed == o.embed && enorm_w == o.enorm_w && hnorm_w == o.hnorm_w && eh_proj == o.eh_proj &&
           final_norm_w == o.final_norm_w && lm_head == o.lm_head && row_scale == o.row_scale &&
           w_dtype == o.w_dtype && tokens_dev == o.tokens_dev && hidden_dev == o.hidden_dev && x_dev == o.x_dev &&
           draft_dev == o.draft_dev && status == o.status && workspace == o.workspace &&
           workspace_bytes == o.workspace_bytes && B == o.B && H == o.H && V == o.V &&
           memcmp(&eps, &o.eps, sizeof(float)) == 0 && stream == o.stream;
  }
};

// Queue one step on s.stream: inputs from tok/hid (host), draft to draft_out, the status word
// to status_out when both it and s.status are given.
int enqueue_host_step(const HostStep& s, const int32_t* tok, const uint16_t* hid, int32_t* draft_out,
                      int32_t* status_out) {
  const size_t hid_bytes = sizeof(uint16_t) * static_cast<size_t>(s.B) * s.H;
  if (cudaMemcpyAsync(s.tokens_dev, tok, sizeof(int32_t) * s.B, cudaMemcpyHostToDevice, s.stream) != cudaSuccess)
    return MTP_ERR_CUDA;
  if (cudaMemcpyAsync(s.hidden_dev, hid, hid_bytes, cudaMemcpyHostToDevice, s.stream) != cudaSuccess)
    return MTP_ERR_CUDA;
  void* cat = s.workspace_bytes >= step_workspace_bytes(s.B, s.H)
                  ? static_cast<uint8_t*>(s.workspace) + step_concat_offset(s.B)
                  : nullptr;
  int v = run_step_input(s.embed, s.enorm_w, s.hnorm_w, s.eh_proj, s.tokens_dev, s.hidden_dev, s.x_dev, s.status,
                         s.B, s.H, s.V, s.eps, s.stream, cat);
  if (v != MTP_OK) return v;
  v = run_output(s.x_dev, s.final_norm_w, s.lm_head, s.row_scale, s.w_dtype, nullptr, s.draft_dev, s.status,
                 s.workspace, s.B, s.H, s.V, s.eps, s.stream);
  if (v != MTP_OK) return v;
  if (cudaMemcpyAsync(draft_out, s.draft_dev, sizeof(int32_t) * s.B, cudaMemcpyDeviceToHost, s.stream) != cudaSuccess)
    return MTP_ERR_CUDA;
  if (s.status && status_out &&
      cudaMemcpyAsync(status_out, s.status, sizeof(int32_t), cudaMemcpyDeviceToHost, s.stream) != cudaSuccess)
    return MTP_ERR_CUDA;
  return MTP_OK;
}

struct StepGraph {
  HostStep key;
  int device = -1;
  std::mutex mu;  // one call at a time uses the staging buffers
  cudaGraphExec_t exec = nullptr;
  int32_t* tok = nullptr;     // pinned staging: [B] tokens, [B, H] hidden, [B] draft, status
  uint16_t* hid = nullptr;
  int32_t* draft = nullptr;
  int32_t* st = nullptr;
  uint32_t* seq = nullptr;    // [0] this call's number, [1] the number the last kernel wrote when done
  uint32_t calls = 0;
  bool polled = false;        // the graph ends in the kernel that writes seq[1]
  uint64_t last_use = 0;
  ~StepGraph() {
    if (exec) cudaGraphExecDestroy(exec);
    if (tok) cudaFreeHost(tok);
  }
};

constexpr size_t kMaxStepGraphs = 8;
std::mutex g_step_mu;
// never destroyed: at process exit the CUDA runtime may already be gone
std::vector<std::shared_ptr<StepGraph>>* g_steps = new std::vector<std::shared_ptr<StepGraph>>();
uint64_t g_step_clock = 0;

// Records the step into a new graph around freshly allocated staging buffers; null on failure
// (the caller then keeps running directly).
std::shared_ptr<StepGraph> record_step(const HostStep& s, int device) {
  auto g = std::make_shared<StepGraph>();
  g->key = s;
  g->device = device;
  const size_t hid_bytes = sizeof(uint16_t) * static_cast<size_t>(s.B) * s.H;
  const size_t tok_bytes = (sizeof(int32_t) * s.B + 15) / 16 * 16;
  uint8_t* base = nullptr;
  if (cudaHostAlloc(reinterpret_cast<void**>(&base), 2 * tok_bytes + 16 + hid_bytes,
                    cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess)
    return nullptr;
  g->tok = reinterpret_cast<int32_t*>(base);
  g->draft = reinterpret_cast<int32_t*>(base + tok_bytes);
  g->st = reinterpret_cast<int32_t*>(base + 2 * tok_bytes);
  g->seq = reinterpret_cast<uint32_t*>(base + 2 * tok_bytes + 8);
  g->seq[0] = g->seq[1] = 0u;
  g->hid = reinterpret_cast<uint16_t*>(base + 2 * tok_bytes + 16);
  // the device's view of the staging buffers: the moves in and out are kernels reading and
  // writing them directly (whole 16-byte pieces of hidden rows); otherwise copy operations
  uint8_t* dbase = nullptr;
  const bool kernel_io = (static_cast<size_t>(s.B) * s.H) % 8 == 0 &&
                         cudaHostGetDevicePointer(reinterpret_cast<void**>(&dbase), base, 0) == cudaSuccess;
  if (!kernel_io) cudaGetLastError();
  if (cudaStreamBeginCapture(s.stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return nullptr;
  int v = MTP_OK;
  if (kernel_io) {
    v = map_cuda(mtp::launch_host_in(reinterpret_cast<const int32_t*>(dbase),
                                     reinterpret_cast<const uint16_t*>(dbase + 2 * tok_bytes + 16), s.tokens_dev,
                                     s.hidden_dev, s.B, s.H, s.stream));
    if (v == MTP_OK) {
      void* cat = s.workspace_bytes >= step_workspace_bytes(s.B, s.H)
                      ? static_cast<uint8_t*>(s.workspace) + step_concat_offset(s.B)
                      : nullptr;
      v = run_step_input(s.embed, s.enorm_w, s.hnorm_w, s.eh_proj, s.tokens_dev, s.hidden_dev, s.x_dev, s.status,
                         s.B, s.H, s.V, s.eps, s.stream, cat);
    }
    // one sequence: the sweep's last CTA writes the draft, the status and the completion word
    // itself; otherwise a small kernel after the sweep does
    bool handed = false;
    if (v == MTP_OK) {
      const mtp::HostBack hb{reinterpret_cast<int32_t*>(dbase + tok_bytes), reinterpret_cast<uint32_t*>(dbase + 2 * tok_bytes)};
      v = map_cuda(mtp::launch_sweep_handback(output_args(s.x_dev, s.final_norm_w, s.lm_head, s.row_scale, s.w_dtype,
                                                          nullptr, s.draft_dev, s.status, s.workspace, s.B, s.H,
                                                          s.V, s.eps),
                                              hb, s.stream, &handed));
    }
    if (v == MTP_OK && !handed)
      v = run_output(s.x_dev, s.final_norm_w, s.lm_head, s.row_scale, s.w_dtype, nullptr, s.draft_dev, s.status,
                     s.workspace, s.B, s.H, s.V, s.eps, s.stream);
    if (v == MTP_OK && !handed)
      v = map_cuda(mtp::launch_host_out(s.draft_dev, reinterpret_cast<int32_t*>(dbase + tok_bytes), s.status,
                                        reinterpret_cast<int32_t*>(dbase + 2 * tok_bytes), s.B,
                                        reinterpret_cast<const uint32_t*>(dbase + 2 * tok_bytes + 8),
                                        reinterpret_cast<uint32_t*>(dbase + 2 * tok_bytes + 12), s.stream));
  } else {
    v = enqueue_host_step(s, g->tok, g->hid, g->draft, g->st);
  }
  cudaGraph_t graph = nullptr;
  const cudaError_t e = cudaStreamEndCapture(s.stream, &graph);
  if (v != MTP_OK || e != cudaSuccess || graph == nullptr) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return nullptr;
  }
  const cudaError_t ei = cudaGraphInstantiate(&g->exec, graph, 0);
  cudaGraphDestroy(graph);
  if (ei != cudaSuccess) {
    g->exec = nullptr;
    cudaGetLastError();
    return nullptr;
  }
  g->polled = kernel_io;
  return g;
}

// Waits for a recorded step that ends in the kernel writing the completion word: polls the word
// (the draft and status are visible once it holds this call's number), and every 4096 polls asks
// the stream, so that a failed launch returns its error and a finished stream ends the wait. This
// avoids the wake-up latency of a stream synchronisation, a few microseconds per step.
int wait_step(const uint32_t* done_word, uint32_t n, cudaStream_t stream) {
  for (uint64_t i = 1;; ++i) {
    if (__atomic_load_n(done_word, __ATOMIC_ACQUIRE) == n) return MTP_OK;
    if ((i & 4095u) == 0) {
      const cudaError_t q = cudaStreamQuery(stream);
      if (q == cudaSuccess) return __atomic_load_n(done_word, __ATOMIC_ACQUIRE) == n ? MTP_OK : MTP_ERR_CUDA;
      if (q != cudaErrorNotReady) return MTP_ERR_CUDA;
    }
  }
}

int run_host_step(const HostStep& s, const int32_t* tokens_host, const uint16_t* hidden_host, int32_t* draft_host) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MTP_ERR_CUDA;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  const bool can_graph = s.stream != nullptr && cudaStreamIsCapturing(s.stream, &cs) == cudaSuccess &&
                         cs == cudaStreamCaptureStatusNone;
  std::shared_ptr<StepGraph> g;
  bool first = false;
  if (can_graph) {
    std::lock_guard<std::mutex> lock(g_step_mu);
    for (auto& e : *g_steps)
      if (e->device == device && e->key.same(s)) g = e;
    first = g == nullptr;
    if (g) g->last_use = ++g_step_clock;
  }
  if (!g) {
    // directly: the caller's host buffers, operation by operation
    int32_t dev_status = 0;
    int v = enqueue_host_step(s, tokens_host, hidden_host, draft_host, &dev_status);
    if (v != MTP_OK) return v;
    if (cudaStreamSynchronize(s.stream) != cudaSuccess) return MTP_ERR_CUDA;
    if (first) {  // everything is initialised now: record the step for the next calls
      std::shared_ptr<StepGraph> rec = record_step(s, device);
      if (rec) {
        std::lock_guard<std::mutex> lock(g_step_mu);
        rec->last_use = ++g_step_clock;
        if (g_steps->size() >= kMaxStepGraphs) {
          size_t lru = 0;
          for (size_t i = 1; i < g_steps->size(); ++i)
            if ((*g_steps)[i]->last_use < (*g_steps)[lru]->last_use) lru = i;
          (*g_steps)[lru] = rec;
        } else {
          g_steps->push_back(rec);
        }
      }
    }
    return s.status ? dev_status : MTP_OK;
  }
  std::lock_guard<std::mutex> lock(g->mu);
  memcpy(g->tok, tokens_host, sizeof(int32_t) * s.B);
  memcpy(g->hid, hidden_host, sizeof(uint16_t) * static_cast<size_t>(s.B) * s.H);
  *g->st = 0;
  uint32_t n = 0;
  if (g->polled) {
    n = ++g->calls;
    if (n == 0) n = ++g->calls;  // 0 is the word's initial value
    __atomic_store_n(&g->seq[0], n, __ATOMIC_RELEASE);
  }
  if (cudaGraphLaunch(g->exec, s.stream) != cudaSuccess) return MTP_ERR_CUDA;
  if (g->polled) {
    const int v = wait_step(&g->seq[1], n, s.stream);
    if (v != MTP_OK) return v;
  } else if (cudaStreamSynchronize(s.stream) != cudaSuccess) {
    return MTP_ERR_CUDA;
  }
  memcpy(draft_host, g->draft, sizeof(int32_t) * s.B);
  return s.status ? *g->st : MTP_OK;
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

int mtp_head_logits_argmax_shard(const uint16_t* x, const uint16_t* final_norm_w, const void* lm_head_shard,
                                 const float* row_scale_shard, int w_dtype, int v0, int n, float* logits,
                                 int64_t* pick, int32_t* draft, int32_t* status, void* workspace,
                                 size_t workspace_bytes, int B, int H, float eps, void* stream) {
  if (!pick) return MTP_ERR_ARG;
  if (v0 < 0 || n < 1 || static_cast<int64_t>(v0) + n > static_cast<int64_t>(INT32_MAX)) return MTP_ERR_SHAPE;
  if (!aligned(pick, 8)) return MTP_ERR_ALIGN;
  const int v = validate_output(x, final_norm_w, lm_head_shard, row_scale_shard, w_dtype, logits, draft, status,
                                workspace, workspace_bytes, B, H, n, eps, /*draft_optional=*/true);
  if (v != MTP_OK) return v;
  return run_output(x, final_norm_w, lm_head_shard, row_scale_shard, w_dtype, logits, draft, status, workspace, B,
                    H, n, eps, stream, v0, pick);
}

int mtp_head_pick_combine(const int64_t* picks, int R, int B, int32_t* draft, float* value, void* stream) {
  if (!picks || !draft) return MTP_ERR_ARG;
  if (R < 1 || R > kMaxPickShards || B < 1 || B > kMaxB) return MTP_ERR_SHAPE;
  if (!aligned(picks, 8) || !aligned(draft, 4) || (value && !aligned(value, 4))) return MTP_ERR_ALIGN;
  return map_cuda(mtp::launch_pick_combine(picks, R, B, draft, value, static_cast<cudaStream_t>(stream)));
}

int64_t mtp_head_pick_key(float value, int32_t index) { return mtp::pick_key(value, index); }

int32_t mtp_head_pick_index(int64_t key) { return mtp::pick_index(key); }

float mtp_head_pick_value(int64_t key) { return mtp::pick_value(key); }

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
  // a workspace of the full size also holds the context-row path's workspace
  void* cat = workspace_bytes >= step_workspace_bytes(B, H) ? static_cast<uint8_t*>(workspace) + step_concat_offset(B)
                                                             : nullptr;
  v = run_step_input(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x, status, B, H, V, eps, stream, cat);
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
  HostStep hs{embed, enorm_w, hnorm_w, eh_proj, final_norm_w, lm_head, row_scale, w_dtype, tokens_dev, hidden_dev,
              x_dev, draft_dev, status, workspace, workspace_bytes, B, H, V, eps, static_cast<cudaStream_t>(stream)};
  return run_host_step(hs, tokens_host, hidden_host, draft_host);
}

int mtp_head_forward_host_args(const mtp_host_step_args* a, const int32_t* tokens_host, const uint16_t* hidden_host,
                               int32_t* draft_host) {
  if (a == nullptr) return MTP_ERR_ARG;
  return mtp_head_forward_host(a->embed, a->enorm_w, a->hnorm_w, a->eh_proj, a->final_norm_w, a->lm_head, a->row_scale,
                               a->w_dtype, tokens_host, hidden_host, a->tokens_dev, a->hidden_dev, a->x_dev,
                               a->draft_dev, draft_host, a->status, a->workspace, a->workspace_bytes, a->B, a->H,
                               a->V, a->eps, a->stream);
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
  const bool have_ws = workspace && workspace_bytes >= mtp::context_workspace_bytes(R, H);
  if (R <= kMaxB && (!have_ws || R == 1 || H % 32 != 0))  // a few rows without room: the batched input stage
    return run_input(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x_out, status, R, H, V, eps, stream);
  if (H % 32 != 0) return MTP_ERR_NOT_IMPLEMENTED;
  if (!have_ws) return MTP_ERR_WORKSPACE;
  return run_context(embed, enorm_w, hnorm_w, eh_proj, tokens, target_hidden, x_out, status, R, H, V, eps, stream,
                     workspace);
}

int mtp_head_quantize_fp8(const uint16_t* w, uint8_t* q, float* row_scale, int32_t* status, int V,
                          int H, void* stream) {
  if (!w || !q || !row_scale || !status) return MTP_ERR_ARG;
  if (check_shape(1, H, V) != MTP_OK) return MTP_ERR_SHAPE;
  if (!aligned(w, 16) || !aligned(q, 16) || !aligned(row_scale, 4) || !aligned(status, 4))
    return MTP_ERR_ALIGN;
  return map_cuda(mtp::launch_quantize(w, q, row_scale, status, V, H, static_cast<cudaStream_t>(stream)));
}

unsigned long long mtp_head_set_wait_limit_ns(unsigned long long ns) { return mtp::set_stage_wait_ns(ns); }

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
