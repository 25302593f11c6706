// Context-row input stage ("glm5next_mtp_head.rs", `rows_impl`: for every context row r the
// embedding row of tokens[r] and hidden row r go through enorm / hnorm, the concat and eh_proj --
// the input stage of `forward_one` per row; the source loops over rows on the host, here all R
// rows run at once).
//
// Two kernels:
//  1. context_concat_kernel: one CTA per row forms the normalised concat [enorm(e_r) | hnorm(h_r)]
//     (the same correctly rounded BF16 values as the single-sequence kernels) into the workspace,
//     plus a flag per row for the token check.
//  2. context_gemm_kernel: x = concat . eh_proj^T, an R x H x 2H GEMM -- compute-bound once R
//     reaches a few hundred rows, so it runs on the fifth-generation tensor cores: 128 x 256
//     output tiles, operands streamed by 2-D TMA tensor loads (128-byte swizzle, the K-major
//     layout the MMA reads directly) into a 4-stage ring, one thread issuing tcgen05.mma
//     (BF16 x BF16, FP32 accumulator in TMEM), one warpgroup moving the accumulator out of TMEM,
//     rounding it to BF16 and storing x. FP32 accumulation is the source's precision for
//     eh_proj.
// Warp roles of the GEMM (256 threads): warp 0 lane 0 = TMA producer, warp 1 = TMEM allocation
// and (lane 0) MMA issue, warps 4..7 = epilogue (warp w reads TMEM lanes 32 (w - 4) ...).
// Every mbarrier wait is bounded; on a timeout the kernel records MTP_ERR_TIMEOUT, still waits
// (bounded) for its own MMAs to finish, frees its TMEM and returns.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/mtp_head.h"
#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace mtp {

namespace {

constexpr int kCtxNormThreads = 512;

// ------------------------------------------------------------------------------- concat
__global__ void __launch_bounds__(kCtxNormThreads) context_concat_kernel(const ContextArgs a) {
  __shared__ float red[2 * (2 * kCtxNormThreads / 32 + 2)];
  __shared__ int ok_s;
  const int r = blockIdx.x;
  const int H = a.H;
  pdl_wait_prior_grid();  // tokens and target_hidden may come from the preceding kernel
  if (threadIdx.x == 0) {
    const int32_t tok = a.tokens[r];
    const int ok = (tok >= 0 && tok < a.V) ? 1 : 0;
    ok_s = ok;
    a.valid[r] = ok;
    if (!ok) store_status(a.status, MTP_ERR_TOKEN_RANGE);
  }
  __syncthreads();
  const bool ok = ok_s != 0;
  uint16_t* c = a.concat + static_cast<size_t>(r) * 2 * H;
  auto job = [&](int j) {
    if (j == 0) {
      const uint16_t* e = ok ? a.embed + static_cast<int64_t>(a.tokens[r]) * H : a.embed;
      return NormJob{e, a.enorm_w, c, ok};
    }
    return NormJob{a.hidden + static_cast<size_t>(r) * H, a.hnorm_w, c + H, true};
  };
  rms_norm_multi_to_smem<kCtxNormThreads>(2, H, a.inv_h, a.eps, red, job, LayoutIdentity{});
  pdl_launch_dependents();
}

// ------------------------------------------------------------------------------- GEMM
constexpr int kGM = 128;                  // output rows (context rows) per tile
constexpr int kGN = 256;                  // output columns (x features) per tile
constexpr int kGK = 64;                   // k elements per stage (one 128-byte swizzle atom)
constexpr int kGStages = 4;
constexpr int kGABytes = kGM * kGK * 2;   // 16 KB
constexpr int kGBBytes = kGN * kGK * 2;   // 32 KB
constexpr int kGStageBytes = kGABytes + kGBBytes;
constexpr int kGThreads = 256;
constexpr uint32_t kTmemCols = kGN;       // FP32 accumulator: 128 lanes x 256 columns

__global__ void __launch_bounds__(kGThreads, 1)
    context_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                        const ContextArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGStages * kGStageBytes);
  uint64_t* empty = full + kGStages;
  uint64_t* acc_full = empty + kGStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kGM, n0 = blockIdx.y * kGN;
  const int K = 2 * a.H;
  const int nkb = K / kGK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kGStages; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), 1);
    }
    mbar_init(smem_addr(acc_full), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), kTmemCols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      pdl_wait_prior_grid();  // the concat comes from the preceding kernel
      const uint64_t pol_b = l2_evict_first_policy();
      uint64_t pol_a;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_a));
      int issued = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kGStages;
        const uint32_t ph = static_cast<uint32_t>(((kb / kGStages) & 1) ^ 1);
        if (*reinterpret_cast<volatile int*>(&abort_flag) || !mbar_wait_bounded(smem_addr(&empty[s]), ph)) {
          store_status(a.status, MTP_ERR_TIMEOUT);
          atomicExch(&abort_flag, 1);
          break;
        }
        const uint32_t bar = smem_addr(&full[s]);
        mbar_arrive_expect_tx(bar, kGStageBytes);
        uint8_t* st = smem + s * kGStageBytes;
        tma_load_2d(smem_addr(st), &tm_a, kb * kGK, m0, bar, pol_a);
        tma_load_2d(smem_addr(st + kGABytes), &tm_b, kb * kGK, n0, bar, pol_b);
        ++issued;
      }
      // every copy issued must land before the CTA's shared memory goes away (normally the
      // MMA thread has already seen them all)
      for (int kb = issued - kGStages < 0 ? 0 : issued - kGStages; kb < issued; ++kb)
        (void)mbar_wait_bounded(smem_addr(&full[kb % kGStages]), static_cast<uint32_t>((kb / kGStages) & 1));
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kGM, kGN);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % kGStages;
        const uint32_t ph = static_cast<uint32_t>((kb / kGStages) & 1);
        if (*reinterpret_cast<volatile int*>(&abort_flag) || !mbar_wait_bounded(smem_addr(&full[s]), ph)) {
          store_status(a.status, MTP_ERR_TIMEOUT);
          atomicExch(&abort_flag, 1);
          break;
        }
        tmem_fence_after_sync();
        const uint32_t sa = smem_addr(smem + s * kGStageBytes);
        const uint64_t da = umma_desc_sw128(sa), db = umma_desc_sw128(sa + kGABytes);
#pragma unroll
        for (int k = 0; k < kGK / 16; ++k)  // 16 elements = 32 bytes along the swizzle row
          umma_bf16(tmem, da + static_cast<uint64_t>((32 * k) >> 4), db + static_cast<uint64_t>((32 * k) >> 4),
                    idesc, (kb | k) != 0 ? 1u : 0u);
        umma_commit(smem_addr(&empty[s]));  // the stage is free once these MMAs have read it
      }
      // always: the epilogue (and the TMEM release) wait for every issued MMA
      umma_commit(smem_addr(acc_full));
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const bool done = mbar_wait_bounded(smem_addr(acc_full), 0);
    tmem_fence_after_sync();
    if (!done) {
      if (lane == 0) store_status(a.status, MTP_ERR_TIMEOUT);
    } else if (!*reinterpret_cast<volatile int*>(&abort_flag)) {
      const int q = warp - 4;  // TMEM lanes 32 q .. 32 q + 31 = tile rows
      const int row = m0 + 32 * q + lane;
      const bool row_ok = row < a.R;
      const bool valid = row_ok && a.valid[row] != 0;
#pragma unroll 1
      for (int c0 = 0; c0 < kGN; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(c0), v);
        if (row_ok && n0 + c0 < a.H) {
          uint16_t* dst = a.x + static_cast<size_t>(row) * a.H + n0 + c0;
          // H is a multiple of 32, so a 32-column slice is inside x or outside it as a whole
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t lo = valid ? bf16_bits_rn(__uint_as_float(v[2 * i])) : 0u;
            const uint32_t hi = valid ? bf16_bits_rn(__uint_as_float(v[2 * i + 1])) : 0u;
            w[i] = lo | (hi << 16);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
      }
    }
  }
  tmem_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    // after a timeout the epilogue may have stopped waiting early: the accumulator is released
    // only once the MMAs issued into it are done (normally this returns at once)
    if (lane == 0) (void)mbar_wait_bounded(smem_addr(acc_full), 0);
    __syncwarp();
    tmem_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
  pdl_launch_dependents();
}

}  // namespace

size_t context_workspace_bytes(int R, int H) {
  const size_t concat = (static_cast<size_t>(R) * 2 * H * 2 + 255) / 256 * 256;
  return concat + static_cast<size_t>(R) * 4;
}

cudaError_t launch_context_rows(const ContextArgs& in, cudaStream_t stream) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  if (in.H % 32 != 0) return cudaErrorNotSupported;
  const TmapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  const size_t smem = 1024 + static_cast<size_t>(kGStages) * kGStageBytes + (2 * kGStages + 1) * 8 + 16;
  if (smem > static_cast<size_t>(di.smem_optin)) return cudaErrorNotSupported;
  ContextArgs a = in;
  const int K = 2 * a.H;
  CUtensorMap ta, tb;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(a.R)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {kGK, kGM};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.concat, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
      return cudaErrorNotSupported;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(a.H)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {kGK, kGN};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.eh_proj), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorNotSupported;
  }
  {
    void* params[] = {&a};
    err = launch_pdl(reinterpret_cast<const void*>(context_concat_kernel), dim3(static_cast<unsigned>(a.R)),
                     dim3(kCtxNormThreads), 0, stream, params);
    if (err != cudaSuccess) return err;
  }
  // output tiles: consecutive CTAs share an eh_proj tile (rows of x tiles run fastest), so each
  // eh_proj tile is read from HBM about once and reused from L2
  const dim3 grid(static_cast<unsigned>((a.R + kGM - 1) / kGM), static_cast<unsigned>((a.H + kGN - 1) / kGN));
  CUtensorMap tac = ta, tbc = tb;
  void* params[] = {&tac, &tbc, &a};
  return launch_pdl(reinterpret_cast<const void*>(context_gemm_kernel), grid, dim3(kGThreads), smem, stream, params);
}

}  // namespace mtp
