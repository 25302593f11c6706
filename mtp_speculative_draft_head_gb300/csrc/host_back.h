// Hand-back of a recorded host-buffer step's result by the single-sequence sweep's last CTA,
// in place of a kernel of its own after the sweep: the step spares that kernel's launch and the
// wait for the sweep's completion before it.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace mtp {

// Device addresses of mapped host memory.
struct HostBack {
  int32_t* draft;   // [1]
  uint32_t* words;  // [0] the status word (when there is one), [2] the call's number, [3] set to [2] last
};

// The output stage of one sequence whose last CTA also writes the draft and the status to hb,
// then, after a system-scope fence, the completion word. *done stays false (nothing launched)
// when the shape does not take the register-resident single-sequence kernel.
cudaError_t launch_sweep_handback(const SweepArgs& a, const HostBack& hb, cudaStream_t stream, bool* done);

}  // namespace mtp
