// Batched input stage on tensor cores: B = 2..16 sequences share one pass over eh_proj
// ("glm5next_mtp_head.rs", `forward_one`: the embedding row at token*hidden, `norm` with enorm
// into concat[0:H] and with hnorm into concat[H:2H], then the `eh_proj` dense gemv n = H,
// k = 2H; here for a batch, as one skinny GEMM  x[B, H] = concat[B, 2H] . eh_proj[H, 2H]^T).
//
// Why not the CUDA-core kernel: that one keeps the sum error-free (TwoSum per product), which
// costs ~8 fp32 operations per product and sequence -- fine for one sequence, but at B = 16 it
// would take ~10x longer than streaming eh_proj. Here the products go through mma.sync
// (m16n8k16, exact BF16 products, FP32 accumulation) over runs of 128 products per output (one
// consumer warp's share of a k-chunk); the run totals are added as double-floats (TwoSum) and x
// is the correctly rounded BF16 of that sum. So x differs from the BF16 of the exact sum only
// where the exact sum lies within the FP32 error of the runs (a few 2^-24 of their absolute
// sums) of a rounding midpoint.
//
// Layout of the work: eh_proj has only H = 6144 rows, too few for 128-row tiles on 152 SMs, so
// every CTA takes a contiguous range of whole 8-row groups (at most 8) and the weights are the
// N operand of the MMA, one group per n-tile; the batch is the M operand (16 sequences, rows
// >= B ignored). No split over k between CTAs, so no workspace and no atomics.
//  * weight producer warp: one 3-D tensor load per stage (8 rows x 1024 elements, 16 KB, L2
//    evict-first, 128-byte swizzle so the ldmatrix reads are bank-conflict free) into a
//    7-stage ring -- few large copies: the same stream in 1 KB row pieces ran at a third of
//    the bandwidth;
//  * activation producer warp: per 1024-element k-chunk, bulk copies of the chunk's part of
//    every embedding row (gathered by token) or target_hidden row and of enorm_w / hnorm_w into
//    a 3-stage ring, so the builders never wait on a global load (a stage is held from its copy
//    through building to its last MMA, so the third stage matters more than an eighth weight
//    stage);
//  * 6 builder warps: turn a stage in place into the normalised concat of all B sequences
//    (rms_norm_vanilla with enorm / hnorm, correctly rounded to BF16 exactly as the
//    single-sequence kernel does);
//  * 8 consumer warps: each owns 8 of the 64 k16-steps of a chunk for every n-tile of the CTA;
//    at the end the 8 double-float partials are added in warp order (deterministic) and
//    rounded once to BF16.
// Prologue (before the first chunk): the 2B sums of squares as double-floats (threads share the
// rows, loads batched), 1/rms in fp64 split into two fp32 parts -- the weights are already in
// flight meanwhile.
// With a caller workspace the concat is instead built once, before this kernel, by the
// row-parallel concat kernel (the same correctly rounded values): every CTA then copies the
// normalised rows and the builders have nothing to do -- at B = 16, normalising all 2B rows in
// each of ~128 CTAs, not the eh_proj stream, had set the time.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace mtp {

namespace {

#ifndef MTP_IN_BUILDERS
#define MTP_IN_BUILDERS 6
#endif
constexpr int kCW = 8;                        // consumer warps
constexpr int kBW = MTP_IN_BUILDERS;          // builder warps
constexpr int kProdWarp = kCW + kBW;          // weight producer warp
constexpr int kActWarp = kProdWarp + 1;       // activation producer warp
constexpr int kInTcThreads = (kCW + kBW + 2) * 32;
constexpr int kPrologueThreads = (kCW + kBW) * 32;
#ifndef MTP_IN_CK
#define MTP_IN_CK 1024
#endif
#ifndef MTP_IN_WSTAGES
#define MTP_IN_WSTAGES (MTP_IN_CK == 512 ? 14 : 7)
#endif
#ifndef MTP_IN_ASTAGES
#define MTP_IN_ASTAGES (MTP_IN_CK == 512 ? 6 : 3)
#endif
#ifndef MTP_IN_FENCE
#define MTP_IN_FENCE 1
#endif
constexpr int kCK = MTP_IN_CK;                // k elements per stage
constexpr int kPitch = kCK * 2 + 16;          // padded row bytes in shared memory
constexpr int kWStageBytes = 8 * kCK * 2;     // one n-tile: 8 weight rows x kCK, 128B-swizzled
constexpr int kWStages = MTP_IN_WSTAGES;
constexpr int kAWOffset = kMaxB * kPitch;     // norm-weight segment after the 16 sequence rows
constexpr int kAStageBytes = kAWOffset + kCK * 2;
constexpr int kAStages = MTP_IN_ASTAGES;
constexpr int kCells = kCK / 8;               // 16-byte cells per sequence row of a chunk
constexpr int kBarInRead = 3;                 // named barrier: prologue has read its inputs
                                              // (prologue -> both producers)
constexpr int kMaxTiles = 8;                  // n-tiles per CTA: at most 64 rows
constexpr int kStepsPerWarp = kCK / 16 / kCW; // k16-steps of a chunk per consumer warp
constexpr int kEpilogueBytes = kCW * kMaxTiles * 32 * 4 * 8;
static_assert(kEpilogueBytes <= kWStages * kWStageBytes, "epilogue scratch reuses the weight ring");
static_assert(kStepsPerWarp % 2 == 0, "the consumer loop takes k16-steps in pairs");

// Byte offset of element k (BF16) of row r (0..7) in a weight stage: the tensor load writes
// [k-block of 64][row][64 elements], each 128-byte row segment swizzled by the row.
__device__ __forceinline__ uint32_t wst_offset(int r, int k) {
  return static_cast<uint32_t>((((k >> 6) * 8 + r) << 7) + ((((k >> 3) & 7) ^ r) << 4));
}

__global__ void __launch_bounds__(kInTcThreads, 1)
    input_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const InputArgs a) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle pattern of the weight stages
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* wring = smem;
  uint8_t* aring = wring + kWStages * kWStageBytes;
  uint64_t* wfull = reinterpret_cast<uint64_t*>(aring + kAStages * kAStageBytes);
  uint64_t* wempty = wfull + kWStages;
  uint64_t* xfull = wempty + kWStages;   // raw activations landed (activation producer)
  uint64_t* afull = xfull + kAStages;     // concat built in place (builders)
  uint64_t* aempty = afull + kAStages;    // concat consumed (consumers)
  float* nrm = reinterpret_cast<float*>(aempty + kAStages);  // [half][sequence][rh, rl]
  DF* part = reinterpret_cast<DF*>(nrm + 2 * kMaxB * 2);       // prologue scratch
  DF* tot = part + kPrologueThreads;
  __shared__ int abort_flag;
  __shared__ int tok_s[kMaxB];
  __shared__ int valid_s[kMaxB];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, K = 2 * H, B = a.B;
  // whole groups of 8 rows per CTA
  const int ngroups = H >> 3;
  const int g0 = static_cast<int>(static_cast<int64_t>(ngroups) * blockIdx.x / gridDim.x);
  const int g1 = static_cast<int>(static_cast<int64_t>(ngroups) * (blockIdx.x + 1) / gridDim.x);
  const int r0 = 8 * g0;
  const int nrows = 8 * (g1 - g0);
  const int ntiles = g1 - g0;
  const int nck = (K + kCK - 1) / kCK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWStages; ++i) {
      mbar_init(smem_addr(&wfull[i]), 1);
      mbar_init(smem_addr(&wempty[i]), kCW);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(smem_addr(&xfull[i]), 1);
      mbar_init(smem_addr(&afull[i]), kBW);
      mbar_init(smem_addr(&aempty[i]), kCW);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kActWarp) {
    // ------------------------------------------------------------------ activation producer
    // Per k-chunk: the chunk's part of every sequence's embedding row (in range tokens only)
    // and target_hidden, and of enorm_w / hnorm_w, copied into the stage the builders then turn
    // into the concat in place.
    asm volatile("bar.sync %0, %1;" ::"r"(kBarInRead), "r"(kPrologueThreads + 64) : "memory");
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      int slot = 0, issued = 0;
      uint32_t ep = 1;
      bool ok = true;
      for (int kc = 0; kc < nck; ++kc) {
        const int k0 = kc * kCK;
        const int k1 = K - k0 < kCK ? K : k0 + kCK;
        const int e1 = k1 < H ? k1 : H;    // embed part: [k0, e1) if k0 < H
        const int h0 = k0 > H ? k0 : H;    // hidden part: [h0, k1) if k1 > H
        const uint32_t eb = k0 < H ? static_cast<uint32_t>(e1 - k0) * 2 : 0u;
        const uint32_t hb = k1 > H ? static_cast<uint32_t>(k1 - h0) * 2 : 0u;
        const uint32_t hoff = static_cast<uint32_t>(h0 - k0) * 2;
        uint32_t bytes = eb + hb;  // the norm-weight segment
        for (int b = 0; b < B; ++b) bytes += (valid_s[b] ? eb : 0u) + hb;
        if (*reinterpret_cast<volatile int*>(&abort_flag) || !mbar_wait_bounded(smem_addr(&aempty[slot]), ep)) {
          ok = false;
          break;
        }
        const uint32_t bar = smem_addr(&xfull[slot]);
        const uint32_t dst = smem_addr(aring + slot * kAStageBytes);
        mbar_arrive_expect_tx(bar, bytes);
        if (eb) bulk_copy_g2s(dst + kAWOffset, a.enorm_w + k0, eb, bar, policy);
        if (hb) bulk_copy_g2s(dst + kAWOffset + hoff, a.hnorm_w + (h0 - H), hb, bar, policy);
        for (int b = 0; b < B; ++b) {
          if (eb && valid_s[b])
            bulk_copy_g2s(dst + b * kPitch, a.embed + static_cast<int64_t>(tok_s[b]) * H + k0, eb, bar, policy);
          if (hb) bulk_copy_g2s(dst + b * kPitch + hoff, a.hidden + static_cast<size_t>(b) * H + (h0 - H), hb, bar, policy);
        }
        ++issued;
        if (++slot == kAStages) { slot = 0; ep ^= 1u; }
      }
      if (!ok) {
        store_status(a.status, MTP_ERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
      for (int s2 = 0; s2 < kAStages && s2 < issued; ++s2) {
        const int uses = (issued - s2 + kAStages - 1) / kAStages;
        (void)mbar_wait_bounded(smem_addr(&xfull[s2]), static_cast<uint32_t>((uses - 1) & 1));
      }
    }
    __syncwarp();
  } else if (warp == kProdWarp) {
    // ------------------------------------------------------------------ weight producer
    // Both streams start once the prologue has read the embedding rows and target_hidden:
    // issued first, ~20 MB of loads over all SMs sit in front of those in the memory queues.
    asm volatile("bar.sync %0, %1;" ::"r"(kBarInRead), "r"(kPrologueThreads + 64) : "memory");
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      int slot = 0, issued = 0;
      uint32_t ep = 1;
      bool ok = true;
      for (int kc = 0; kc < nck && ok; ++kc) {
        for (int t = 0; t < ntiles; ++t) {
          if (*reinterpret_cast<volatile int*>(&abort_flag) || !mbar_wait_bounded(smem_addr(&wempty[slot]), ep)) {
            ok = false;
            break;
          }
          // one tensor load: 8 rows x kCK elements (k-blocks past the row end read as zeros)
          const uint32_t bar = smem_addr(&wfull[slot]);
          mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kWStageBytes));
          tma_load_3d(smem_addr(wring + slot * kWStageBytes), &tmap_w, 0, r0 + 8 * t, kc * (kCK / 64), bar, policy);
          ++issued;
          if (++slot == kWStages) { slot = 0; ep ^= 1u; }
        }
      }
      if (!ok) {
        store_status(a.status, MTP_ERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
      // every copy issued must land before the CTA's shared memory goes away
      for (int s = 0; s < kWStages && s < issued; ++s) {
        const int uses = (issued - s + kWStages - 1) / kWStages;
        (void)mbar_wait_bounded(smem_addr(&wfull[s]), static_cast<uint32_t>((uses - 1) & 1));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ prologue (warps 0..11)
    pdl_wait_prior_grid();  // tokens and target_hidden may come from the preceding kernel
    if (threadIdx.x < B) {
      const int32_t tok = a.tokens[threadIdx.x];
      const bool ok = tok >= 0 && tok < a.V;
      valid_s[threadIdx.x] = ok ? 1 : 0;
      tok_s[threadIdx.x] = ok ? tok : 0;
      if (!ok) store_status(a.status, MTP_ERR_TOKEN_RANGE);
    }
    named_barrier_sync(1, kPrologueThreads);
    {
      auto row = [&](int j) -> const uint16_t* {
        const int b = j >> 1;
        if (j & 1) return a.hidden + static_cast<size_t>(b) * H;
        return valid_s[b] ? a.embed + static_cast<int64_t>(tok_s[b]) * H : nullptr;
      };
      sumsq_rows<kPrologueThreads, 8, false>(2 * B, H, row, nullptr, part, nullptr, tot, nullptr, 1);
      asm volatile("bar.arrive %0, %1;" ::"r"(kBarInRead), "r"(kPrologueThreads + 64) : "memory");
      if (threadIdx.x < 2 * B) {
        const int b = threadIdx.x >> 1, half = threadIdx.x & 1;
        const DF t = tot[threadIdx.x];
        // 1 / rms in fp64 (rsqrt: within an ulp or two of the correctly rounded value)
        const double ms = (static_cast<double>(t.hi) + static_cast<double>(t.lo)) * a.inv_h;
        const double rr = rsqrt(ms + static_cast<double>(a.eps));
        const float rh = static_cast<float>(rr);
        nrm[(half * kMaxB + b) * 2] = rh;
        nrm[(half * kMaxB + b) * 2 + 1] = static_cast<float>(rr - static_cast<double>(rh));
      }
    }
    named_barrier_sync(1, kPrologueThreads);
    pdl_launch_dependents();

    if (warp >= kCW) {
      // ---------------------------------------------------------------- builders
      // The stage holds the raw BF16 inputs of this chunk (row b: embedding / target_hidden
      // segment; then the norm-weight segment); each 8-element piece is replaced in place by its
      // normalised, correctly rounded concat values.
      // thread -> 16-byte cells bt, bt + 32 * kBW, ... of the chunk (sequence-major)
      const int bt = threadIdx.x - kCW * 32;
      int slot = 0;
      uint32_t xp = 0;
      for (int kc = 0; kc < nck; ++kc) {
        const int k0 = kc * kCK;
        const int ppr = (K - k0 < kCK ? K - k0 : kCK) >> 3;  // 8-element pieces per sequence
        if (*reinterpret_cast<volatile int*>(&abort_flag) ||
            !__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&xfull[slot]), xp))) {
          if (lane == 0) {
            store_status(a.status, MTP_ERR_TIMEOUT);
            atomicExch(&abort_flag, 1);
          }
          break;
        }
        uint8_t* base = aring + slot * kAStageBytes;
        for (int cell = bt; cell < B * kCells; cell += kBW * 32) {
          const int b = cell / kCells, c = cell - b * kCells;
          if (c < ppr) {
            const int half = k0 + 8 * c >= H ? 1 : 0;
            uint4* cp = reinterpret_cast<uint4*>(base + b * kPitch + c * 16);
            uint4 o = make_uint4(0u, 0u, 0u, 0u);
            if (half || valid_s[b]) {
              const uint4 wq = *reinterpret_cast<const uint4*>(base + kAWOffset + c * 16);
              const float wf[8] = {bf16_lo(wq.x), bf16_hi(wq.x), bf16_lo(wq.y), bf16_hi(wq.y),
                                   bf16_lo(wq.z), bf16_hi(wq.z), bf16_lo(wq.w), bf16_hi(wq.w)};
              const uint4 xq = *cp;
              const uint32_t xu[4] = {xq.x, xq.y, xq.z, xq.w};
              o = bf16x8_scaled_rne(xu, wf, nrm[(half * kMaxB + b) * 2], nrm[(half * kMaxB + b) * 2 + 1]);
            }
            *cp = o;
          }
        }
        fence_proxy_async_smem();  // the stage is refilled by bulk copies once consumed
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&afull[slot]));
        if (++slot == kAStages) { slot = 0; xp ^= 1u; }
      }
    } else {
      // ---------------------------------------------------------------- consumers
      // Per chunk and n-tile the warp's MMAs (kStepsPerWarp * 16 products per output) start from
      // zero; each chunk total then goes into a double-float with TwoSum, so the only rounding
      // left in x before the final one is that of these short tensor-core sums.
      DF xs[kMaxTiles][4];
#pragma unroll
      for (int t = 0; t < kMaxTiles; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) xs[t][i] = DF{0.0f, 0.0f};
      int wslot = 0, aslot = 0;
      uint32_t wp = 0, ap = 0;
      bool ok = true;
      for (int kc = 0; kc < nck && ok; ++kc) {
        const int k0 = kc * kCK;
        const int nks = (K - k0 < kCK ? K - k0 : kCK) >> 4;  // k16-steps in this chunk
        int mine = nks - kStepsPerWarp * warp;  // this warp's steps: kStepsPerWarp * w + 0, 1, ...
        mine = mine < 0 ? 0 : (mine > kStepsPerWarp ? kStepsPerWarp : mine);
        if (*reinterpret_cast<volatile int*>(&abort_flag) ||
            !__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&afull[aslot]), ap))) {
          ok = false;
          break;
        }
        const uint32_t abase = smem_addr(aring + aslot * kAStageBytes);
        uint32_t af[kStepsPerWarp][4];
#pragma unroll
        for (int s = 0; s < kStepsPerWarp; ++s) {
          if (s < mine) {
            const int kk = (kStepsPerWarp * warp + s) * 16 + 8 * (lane >> 4);
            ldmatrix_x4(af[s], abase + (lane & 15) * kPitch + kk * 2);
          }
        }
#pragma unroll
        for (int t = 0; t < kMaxTiles; ++t) {
          if (t < ntiles && ok) {
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&wfull[wslot]), wp))) {
              ok = false;
            } else {
              const uint32_t wbase = smem_addr(wring + wslot * kWStageBytes);
              float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
              for (int sp = 0; sp < kStepsPerWarp / 2; ++sp) {
                if (2 * sp < mine) {
                  uint32_t bf[4];
                  const int kk = (kStepsPerWarp * warp + 2 * sp) * 16 + 8 * (lane >> 3);
                  ldmatrix_x4(bf, wbase + wst_offset(lane & 7, kk));
                  mma_bf16(c, af[2 * sp], bf[0], bf[1]);
                  if (2 * sp + 1 < mine) mma_bf16(c, af[2 * sp + 1], bf[2], bf[3]);
                }
              }
              if (MTP_IN_FENCE) fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) mbar_arrive(smem_addr(&wempty[wslot]));
              if (++wslot == kWStages) { wslot = 0; wp ^= 1u; }
#pragma unroll
              for (int i = 0; i < 4; ++i) df_add(xs[t][i], c[i]);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&aempty[aslot]));
        if (++aslot == kAStages) { aslot = 0; ap ^= 1u; }
      }
      if (!ok && lane == 0) {
        store_status(a.status, MTP_ERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
      // All weight stages consumed (so no copy is in flight): the ring becomes the scratch of the
      // cross-warp sum, [warp][n-tile][lane][4] double-floats. Both barriers are unconditional;
      // after the first one the flag no longer changes (every stage was produced and built, or
      // some consumer warp has already set it).
      named_barrier_sync(2, kCW * 32);
      const bool aborted = *reinterpret_cast<volatile int*>(&abort_flag) != 0;
      float2* red = reinterpret_cast<float2*>(wring);
      if (!aborted) {
#pragma unroll
        for (int t = 0; t < kMaxTiles; ++t)
          if (t < ntiles)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[((warp * kMaxTiles + t) * 32 + lane) * 4 + i] = make_float2(xs[t][i].hi, xs[t][i].lo);
      }
      named_barrier_sync(2, kCW * 32);
      if (!aborted) {
        for (int o = threadIdx.x; o < B * nrows; o += kCW * 32) {
          const int b = o / nrows, rloc = o - b * nrows;
          const int t = rloc >> 3, n = rloc & 7;
          // C fragment: lane 4g + q holds (m = g, n = 2q, 2q+1) in c0, c1 and (m = g + 8, ...) in c2, c3
          const int ln = 4 * (b & 7) + (n >> 1), i = 2 * (b >> 3) + (n & 1);
          const float2 v0 = red[(t * 32 + ln) * 4 + i];
          DF tot{v0.x, v0.y};
#pragma unroll
          for (int w = 1; w < kCW; ++w) {
            const float2 v = red[((w * kMaxTiles + t) * 32 + ln) * 4 + i];
            tot = df_add(tot, DF{v.x, v.y});
          }
          // an out-of-range token gives an all-zero x row (and the status set in the prologue)
          a.x[static_cast<size_t>(b) * H + r0 + rloc] = valid_s[b] ? bf16_rne_df(tot.hi, tot.lo) : uint16_t(0);
        }
      }
    }
  }
}

}  // namespace

size_t input_tc_smem_bytes() {
  return 1024 + static_cast<size_t>(kWStages) * kWStageBytes + static_cast<size_t>(kAStages) * kAStageBytes +
         (2 * kWStages + 3 * kAStages) * 8 + 2 * kMaxB * 2 * sizeof(float) +
         (kPrologueThreads + 2 * kMaxB) * sizeof(DF) + 128;
}

cudaError_t launch_input_tc(const InputArgs& a, cudaStream_t stream, bool* launched) {
  *launched = false;
  // rows of 2H elements must split into whole 64-element k-blocks for the tensor map
  if (a.B < 2 || a.B > kMaxB || a.H % 32 != 0) return cudaSuccess;
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  const size_t smem = input_tc_smem_bytes();
  if (smem > static_cast<size_t>(di.smem_optin)) return cudaSuccess;
  const TmapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaSuccess;
  // eh_proj [H, 2H] viewed as [2H / 64 k-blocks][H rows][64 elements]: a box of 8 rows x
  // kCK / 64 k-blocks is one weight stage, 128-byte swizzled
  const int K = 2 * a.H;
  CUtensorMap tm;
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(a.H), static_cast<cuuint64_t>(K / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
  const cuuint32_t box[3] = {64, 8, static_cast<cuuint32_t>(kCK / 64)};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a.eh_proj), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaSuccess;
  // whole 8-row groups per CTA, at most kMaxTiles; the grid is the smallest one with the
  // fewest groups on any CTA
  const int64_t ngroups = a.H / 8;
  int64_t grid = di.sm_count < ngroups ? di.sm_count : ngroups;
  int64_t per = (ngroups + grid - 1) / grid;
  if (per > kMaxTiles) per = kMaxTiles;
  grid = (ngroups + per - 1) / per;
  InputArgs args = a;
  CUtensorMap tmc = tm;
  void* params[] = {&tmc, &args};
  *launched = true;
  return launch_pdl(reinterpret_cast<const void*>(input_tc_kernel), dim3(static_cast<unsigned>(grid)),
                    dim3(kInTcThreads), smem, stream, params);
}

}  // namespace mtp
