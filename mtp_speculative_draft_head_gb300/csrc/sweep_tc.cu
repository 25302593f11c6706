// Batched output stage on tensor cores: B = 2..16 sequences share one pass over lm_head
// ("glm5next_mtp_head.rs", `forward_one`: shared_head.norm, the lm_head gemv, argmax; here for a
// batch, as one skinny GEMM  logits[B, V] = xhat[B, H] . lm_head[V, H]^T  fused with the argmax).
//
// Why tensor cores here and not at B = 1: per weight byte the batch needs B multiply-adds, which
// past B ~ 2-4 outruns the fp32 FMA issue rate while HBM still has bandwidth to spare. The need is
// modest (a 16-sequence BF16 sweep at the HBM roofline is ~110 TFLOP/s, FP8 ~220), so warp-level
// mma.sync (m16n8k16, FP32 accumulation) covers it with register operands -- which lets FP8 codes
// be widened straight into A fragments by the hardware E4M3 -> f16 conversion, with no trip
// through shared memory.
//
// Roles (384 threads, 12 warps: up to 168 registers a thread):
//  * producer warp: streams 128-row tiles of lm_head, two 128-byte k-blocks per row and stage,
//    with 2-D TMA tensor loads (128-byte swizzle) into a 6-stage ring of 32 KB (mbarrier
//    full/empty pairs, bounded waits);
//  * 3 builder warps: compute xhat = rms_norm_vanilla(x, final_norm_w) one stage at a time
//    (BF16 for a BF16 head; for FP8, f16 scaled by 2^k per sequence, exact) into a small ring, in
//    the same swizzled layout, with the same exact rounding as the other kernels. The sums of
//    squares behind 1/rms come from a small kernel launched just before (xnorm_parts_kernel);
//  * 8 consumer warps: 16 rows each of a 128-row tile; ldmatrix + mma.sync, batch as N (8 or 16).
// Loop order: groups of 4 row tiles; per stage the activations are built once and used by every
// tile of the group, whose accumulators stay in registers. Each lm_head byte is read once.
// FP8 A fragments come out of ldmatrix with four codes per register; with k permuted the same way
// in the activations (codes 4t..4t+3 of a 16-code block sit in k slots 2t, 2t+1, 2t+8, 2t+9 of
// thread t) every product pairs the right code with the right activation.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace mtp {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kBuilderWarps = 3;
constexpr int kTcWarps = kConsumerWarps + kBuilderWarps + 1;
constexpr int kTcThreads = kTcWarps * 32;          // 384: three warps per SM sub-partition, so
                                                   // up to 168 registers a thread
constexpr int kPrologueThreads = (kConsumerWarps + kBuilderWarps) * 32;  // 352
constexpr int kTileRows = 16 * kConsumerWarps;     // 128
// Row tiles per group (their accumulators stay in registers while the activations of a stage
// are reused across them). Four: with two n-tiles (B > 8) the FP8 activation fragments of a
// stage take 64 registers, and measured at H = 6144, V = 154880 groups of 4 were also ~4 us
// faster than groups of 8 for every other batch and weight type (B = 4, 8: BF16 284 -> 280 us,
// FP8 153 -> 149 us).
template <int WT, int NT>
__host__ __device__ constexpr int tile_group() { return 4; }
constexpr int kATileBytes = kTileRows * 128;       // 16 KB: 128 rows x 128 bytes (one k-block)
// A weight stage holds kKS consecutive k-blocks of one row tile (two tensor loads issued back to
// back): each row is then read 256 contiguous bytes at a time. With one k-block per visit (128
// bytes per row, the next 128 bytes only after the group's other 1023 rows) the same stream
// reached 78% of the HBM bandwidth instead of 95%.
constexpr int kKS = 2;
constexpr int kAStageBytes = kKS * kATileBytes;    // 32 KB
constexpr int kAStages = 6;
constexpr int kSeq = 16;                           // activation rows per B tile (N <= 16)
constexpr int kProducerWarp = kConsumerWarps + kBuilderWarps;

template <int WT>
struct TcCfg {
  static constexpr int kKbElems = (WT == MTP_W_BF16) ? 64 : 128;  // weights per row per k-block
  static constexpr int kBTileBytes = kSeq * kKbElems * 2;         // bf16 / f16 activations
  static constexpr int kBStageBytes = kKS * kBTileBytes;
  static constexpr int kBStages = (WT == MTP_W_BF16) ? 4 : 3;
};

// ---------------------------------------------------------------------------- MMA of one stage
// The activation (B-operand) fragments of a k-block are the same for every row tile of a group:
// they are loaded into registers once per k-block (and the activation stage released at once).
template <int WT, int NT>
struct BFrags;

// BF16 head: k-block of 64, four k16-steps; fragment (b0, b1) per step and n-tile.
template <int NT>
struct BFrags<MTP_W_BF16, NT> {
  uint32_t r[4][NT][2];
  __device__ __forceinline__ void load(uint32_t b_base, int lane) {
    const int bn = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if constexpr (NT == 2) {
        uint32_t b[4];
        ldmatrix_x4(b, b_base + swz(bn, 2 * kk + ((lane >> 3) & 1)));
        r[kk][0][0] = b[0]; r[kk][0][1] = b[1]; r[kk][1][0] = b[2]; r[kk][1][1] = b[3];
      } else {
        uint32_t b[2];
        ldmatrix_x2(b, b_base + swz(lane & 7, 2 * kk + ((lane >> 3) & 1)));
        r[kk][0][0] = b[0]; r[kk][0][1] = b[1];
      }
    }
  }
  // A = this warp's 16 rows x 64 k of a 128-row tile
  __device__ __forceinline__ void mma(uint32_t a_base, float (&acc)[NT][4], int warp, int lane) const {
    const int ar = 16 * warp + (lane & 15);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      ldmatrix_x4(a, a_base + swz(ar, 2 * kk + (lane >> 4)));
#pragma unroll
      for (int jn = 0; jn < NT; ++jn) mma_bf16(acc[jn], a, r[kk][jn][0], r[kk][jn][1]);
    }
  }
};

// FP8 head: k-block of 128 codes, eight k16-steps over two 64-element activation sub-tiles.
// ldmatrix hands each thread four consecutive codes (4*t4 .. 4*t4+3 of a 16-code block); they
// fill k slots 2*t4, 2*t4+1, 2*t4+8, 2*t4+9 of the MMA, so the activation fragment of that
// thread is x[4*t4 .. 4*t4+3] of the same block -- one 8-byte load.
template <int NT>
struct BFrags<MTP_W_FP8_E4M3, NT> {
  uint32_t r[8][NT][2];
  __device__ __forceinline__ void load(uint32_t b_base, int lane) {
    const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const int kin = 16 * s + 4 * t4;  // code offset within the 128-code block
      const int st = kin >> 6, ke = kin & 63;
#pragma unroll
      for (int jn = 0; jn < NT; ++jn)
        lds_v2(r[s][jn][0], r[s][jn][1], b_base + st * 2048 + swz(8 * jn + g, ke >> 3) + ((ke & 7) << 1));
    }
  }
  __device__ __forceinline__ void mma(uint32_t a_base, float (&acc)[NT][4], int warp, int lane) const {
    const int ar = 16 * warp + (lane & 15);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t c[4];
      ldmatrix_x4(c, a_base + swz(ar, 2 * q + (lane >> 4)));
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t a[4];
        e4m3x4_to_f16x2x2(c[2 * h], a[0], a[2]);      // row g:   codes 4t4, 4t4+1 | 4t4+2, 4t4+3
        e4m3x4_to_f16x2x2(c[2 * h + 1], a[1], a[3]);  // row g+8
#pragma unroll
        for (int jn = 0; jn < NT; ++jn) mma_f16(acc[jn], a, r[2 * q + h][jn][0], r[2 * q + h][jn][1]);
      }
    }
  }
};

// CTA combine of per-warp bests (wbest[warp * kSeq + b]) and the last-CTA-done grid argmax.
__device__ void tc_argmax_finish(int nb, const ArgBest* wbest, const SweepArgs& a) {
  uint8_t* ws = a.ws;
  __shared__ int is_last;
  unsigned int* counter = reinterpret_cast<unsigned int*>(ws);
  if (threadIdx.x < nb) {
    ArgBest c{0.0f, -1};
    for (int w = 0; w < kTcWarps; ++w) {
      const ArgBest o = wbest[w * kSeq + threadIdx.x];
      if (o.i >= 0) arg_update(c, o.v, o.i);
    }
    pick_publish(ws, threadIdx.x, c.v, c.i, a.index_base);
    __threadfence();
  }
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(counter, 1u) == gridDim.x - 1) ? 1 : 0;
  __syncthreads();
  if (is_last) {
    __threadfence();
    if (threadIdx.x < nb) pick_finish(ws, threadIdx.x, a.draft, a.pick);
    if (threadIdx.x == 0) atomicExch(counter, 0u);
  }
}

// ---------------------------------------------------------------------------- norm parts
// The sums of squares behind shared_head.norm's 1/rms (and, for an FP8 head, max |x w_f|, which
// fixes the power-of-two scale of the f16 activations) of every row of x, computed once per call
// instead of in each of the sweep's CTAs: there, every CTA summed all B rows itself, 152 times
// the same double-float work, ~9 us of the sweep at B = 16. One warp per slice of a row
// (grid kNormParts x B); each writes {sum hi, sum lo, max, 0} to the workspace header, and the
// sweep adds a row's kNormParts slices in order. At most 32 registers a thread and no shared
// memory, so a CTA of it fits on an SM beside a running sweep CTA (which leaves ~1000 registers
// free): it starts while the kernel before is still finishing and never keeps a sweep CTA off
// its SM. Measured at H = 6144 (one GB300, 50-launch CUDA graphs), the same drafts: the FP8
// sweep at B = 16 from 165.5 to 160.3 us, BF16 from 298.5 to 290.6 us, and the whole batched
// step 205 -> 199.7 us (FP8) and 333 -> 325.7 us (BF16). A version with 256-thread CTAs was
// slower for the sweep alone (FP8 B = 16: 165 -> 168.6 us): its CTAs kept 16 SMs from the sweep
// for their run, and those SMs' CTAs finished last.
template <int WT>
__global__ void __maxnreg__(32) xnorm_parts_kernel(const SweepArgs a) {
  const int p = blockIdx.x, b = blockIdx.y, lane = threadIdx.x, H = a.H;
  // the sweep may launch at once: its CTAs wait for this grid before they read the parts
  pdl_launch_dependents();
  pdl_wait_prior_grid();  // x comes from the preceding kernel
  const int nv = H >> 3;  // 16-byte vectors of a row
  const int v0 = static_cast<int>(static_cast<int64_t>(nv) * p / kNormParts);
  const int v1 = static_cast<int>(static_cast<int64_t>(nv) * (p + 1) / kNormParts);
  const uint4* xv = reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(b) * H);
  const uint4* wv = reinterpret_cast<const uint4*>(a.final_norm_w);
  DF acc{0.0f, 0.0f};
  float mx = 0.0f;
#pragma unroll 3
  for (int v = v0 + lane; v < v1; v += 32) {
    const uint4 q = xv[v];
    const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float lo = bf16_lo(u[t]), hi = bf16_hi(u[t]);
      df_add(acc, __fmul_rn(lo, lo));  // squares of BF16 values are exact in fp32
      df_add(acc, __fmul_rn(hi, hi));
    }
    if constexpr (WT == MTP_W_FP8_E4M3) {
      const uint4 wq = wv[v];
      const uint32_t w4[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        mx = fmaxf(mx, fabsf(__fmul_rn(bf16_lo(u[t]), bf16_lo(w4[t]))));
        mx = fmaxf(mx, fabsf(__fmul_rn(bf16_hi(u[t]), bf16_hi(w4[t]))));
      }
    }
  }
  // fixed butterfly: the result does not depend on timing
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) {
    acc = df_add(acc, shfl_xor_df(acc, m));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
  }
  if (lane == 0)
    reinterpret_cast<float4*>(a.ws + kWsNormOffset)[b * kNormParts + p] = make_float4(acc.hi, acc.lo, mx, 0.0f);
}

// ---------------------------------------------------------------------------- the kernel
template <int WT, int NT>
__global__ void __launch_bounds__(kTcThreads, 1)
    sweep_tc_kernel(const __grid_constant__ CUtensorMap tmap_w, const SweepArgs a) {
  using Cfg = TcCfg<WT>;
  constexpr int kTileGroup = tile_group<WT, NT>();
  constexpr int KBE = Cfg::kKbElems;
  constexpr int BTB = Cfg::kBTileBytes;     // activations of one k-block
  constexpr int BSB = Cfg::kBStageBytes;    // one activation stage (kKS k-blocks)
  constexpr int kBStages = Cfg::kBStages;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle pattern
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* aring = smem;
  uint8_t* bring = aring + kAStages * kAStageBytes;
  uint64_t* afull = reinterpret_cast<uint64_t*>(bring + kBStages * BSB);
  uint64_t* aempty = afull + kAStages;
  uint64_t* bfull = aempty + kAStages;
  uint64_t* bempty = bfull + kBStages;
  float* nrm = reinterpret_cast<float*>(bempty + kBStages);  // rh, rl, xscale, unscale [4][16]
  ArgBest* wbest = reinterpret_cast<ArgBest*>(nrm + 4 * kSeq);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.B, H = a.H;
  const int64_t V = a.V;
  const int KB = (H + KBE - 1) / KBE;
  const int KP = (KB + kKS - 1) / kKS;  // weight / activation stages per row tile
  const int T = static_cast<int>((V + kTileRows - 1) / kTileRows);
  const int t0 = static_cast<int>(static_cast<int64_t>(T) * blockIdx.x / gridDim.x);
  const int t1 = static_cast<int>(static_cast<int64_t>(T) * (blockIdx.x + 1) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(smem_addr(&afull[i]), 1);
      mbar_init(smem_addr(&aempty[i]), kConsumerWarps);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(smem_addr(&bfull[i]), kBuilderWarps);
      mbar_init(smem_addr(&bempty[i]), kConsumerWarps);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  for (int i = threadIdx.x; i < kTcWarps * kSeq; i += kTcThreads) wbest[i] = ArgBest{0.0f, -1};
  __syncthreads();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ producer
    // lm_head does not depend on the kernels before: the weight stream starts at once, while
    // the prologue waits for the norm parts. (When the prologue itself summed the squares of
    // all of x, the stream had to wait for those reads: ~30 MB of tensor loads in front of them
    // in the memory queues delayed them by several microseconds.)
    int issued = 0;
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      int slot = 0;
      uint32_t ep = 1;
      bool ok = true;
      for (int gt = t0; gt < t1 && ok; gt += kTileGroup) {
        const int ntile = (t1 - gt) < kTileGroup ? (t1 - gt) : kTileGroup;
        for (int kp = 0; kp < KP && ok; ++kp) {
          const int nsub = KB - kp * kKS < kKS ? KB - kp * kKS : kKS;
          for (int j = 0; j < ntile; ++j) {
            if (*reinterpret_cast<volatile int*>(&abort_flag) || !mbar_wait_bounded(smem_addr(&aempty[slot]), ep, a.wait_ns)) {
              ok = false;
              break;
            }
            const uint32_t bar = smem_addr(&afull[slot]);
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nsub * kATileBytes));
            for (int sb = 0; sb < nsub; ++sb)
              tma_load_2d(smem_addr(aring + slot * kAStageBytes + sb * kATileBytes), &tmap_w, (kp * kKS + sb) * KBE,
                          (gt + j) * kTileRows, bar, policy);
            ++issued;
            if (++slot == kAStages) { slot = 0; ep ^= 1u; }
          }
        }
      }
      if (!ok) {
        store_status(a.status, MTP_ERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
      // every copy issued must land before the CTA's shared memory goes away
      for (int s = 0; s < kAStages && s < issued; ++s) {
        const int uses = (issued - s + kAStages - 1) / kAStages;
        (void)mbar_wait_bounded(smem_addr(&afull[s]), static_cast<uint32_t>((uses - 1) & 1));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ prologue (warps 0..11)
    pdl_wait_prior_grid();  // the norm parts (and x) come from the preceding kernels
    {
      if (threadIdx.x < B) {
        const int b = threadIdx.x;
        // a row's slices in order: the sum does not depend on timing
        const float4* pp = reinterpret_cast<const float4*>(a.ws + kWsNormOffset) + b * kNormParts;
        DF tot{0.0f, 0.0f};
        float mtot = 0.0f;
#pragma unroll
        for (int q = 0; q < kNormParts; ++q) {  // all eight loads in flight at once
          const float4 v = __ldcg(pp + q);
          tot = df_add(tot, DF{v.x, v.y});
          mtot = fmaxf(mtot, v.z);
        }
        // 1 / rms in fp64 (rsqrt: within an ulp or two of the correctly rounded value)
        const double ms = (static_cast<double>(tot.hi) + static_cast<double>(tot.lo)) * a.inv_h;
        const double rr = rsqrt(ms + static_cast<double>(a.eps));
        const float rh = static_cast<float>(rr);
        const float rl = static_cast<float>(rr - static_cast<double>(rh));
        nrm[b] = rh;
        nrm[kSeq + b] = rl;
        float xs = 1.0f, us = 1.0f;
        if constexpr (WT == MTP_W_FP8_E4M3) {
          // largest |xhat| of this sequence: rounding is monotonic, so it is the rounded max
          const float mx = mtot;
          const float yh = __fmul_rn(mx, rh);
          const float yl = __fmaf_rn(mx, rl, __fmaf_rn(mx, rh, -yh));
          const float m = bf16_bits_to_f32(bf16_rne_df(yh, yl));
          if (m > 0.0f && m <= 3.0e38f) {
            int e = 0;
            (void)frexpf(m, &e);
            xs = ldexpf(1.0f, 15 - e);
            us = ldexpf(1.0f, e - 15);
          }
        }
        nrm[2 * kSeq + b] = xs;
        nrm[3 * kSeq + b] = us;
      }
    }
    pdl_launch_dependents();

    if (warp >= kConsumerWarps) {
      // ---------------------------------------------------------------- builders
      // A sub-tile has 16 sequences x 8 cells of 16 bytes; this thread's cells are bt, bt + 96.
      // The stages follow one another over the groups (u = group * KP + kp); the x / weight
      // vectors of stage u + 1 are loaded into registers as soon as stage u is published, so
      // their latency overlaps the wait for the next free slot.
      constexpr int kSubs = BSB / 2048;
      constexpr int kCellIt = (kSeq * 8 + kBuilderWarps * 32 - 1) / (kBuilderWarps * 32);
      const int bt = threadIdx.x - kConsumerWarps * 32;  // 0..95
      const int ngroups = (t1 - t0 + kTileGroup - 1) / kTileGroup;
      const int nstages = ngroups * KP;
      uint4 xr[kSubs][kCellIt], wr[kSubs][kCellIt];
      auto fetch = [&](int u) {
        const int kp = u % KP;
#pragma unroll
        for (int sub = 0; sub < kSubs; ++sub)
#pragma unroll
          for (int ci = 0; ci < kCellIt; ++ci) {
            const int cell = bt + ci * kBuilderWarps * 32;
            const int n = cell >> 3, c = cell & 7;
            const int k0 = kp * kKS * KBE + 64 * sub + 8 * c;
            if (cell < kSeq * 8 && n < B && k0 < H) {
              xr[sub][ci] = *reinterpret_cast<const uint4*>(a.x + static_cast<size_t>(n) * H + k0);
              wr[sub][ci] = *reinterpret_cast<const uint4*>(a.final_norm_w + k0);
            }
          }
      };
      // x and w_f of the first stage are on their way before the wait for the norm factors
      // (0.5 to 1.4 us off a batched sweep or step, measured)
      if (nstages > 0) fetch(0);
      named_barrier_sync(1, kPrologueThreads);  // the norm factors are in `nrm`
      int slot = 0;
      uint32_t ep = 1;
      for (int u = 0; u < nstages; ++u) {
        const int kp = u % KP;
        if (*reinterpret_cast<volatile int*>(&abort_flag) ||
            !__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&bempty[slot]), ep, a.wait_ns))) {
          if (lane == 0) {
            store_status(a.status, MTP_ERR_TIMEOUT);
            atomicExch(&abort_flag, 1);
          }
          break;
        }
        uint8_t* bt_base = bring + slot * BSB;
        // 2 KB sub-tiles of 64 activations x 16 sequences, k-block-major (zeros past H)
#pragma unroll
        for (int sub = 0; sub < kSubs; ++sub)
#pragma unroll
          for (int ci = 0; ci < kCellIt; ++ci) {
            const int cell = bt + ci * kBuilderWarps * 32;
            const int n = cell >> 3, c = cell & 7;
            const int k0 = kp * kKS * KBE + 64 * sub + 8 * c;
            if (cell < kSeq * 8) {
              uint4 o = make_uint4(0u, 0u, 0u, 0u);
              if (n < B && k0 < H) {
                const uint4 xq = xr[sub][ci], wq = wr[sub][ci];
                const uint32_t xu[4] = {xq.x, xq.y, xq.z, xq.w};
                const float wf[8] = {bf16_lo(wq.x), bf16_hi(wq.x), bf16_lo(wq.y), bf16_hi(wq.y),
                                     bf16_lo(wq.z), bf16_hi(wq.z), bf16_lo(wq.w), bf16_hi(wq.w)};
                o = bf16x8_scaled_rne(xu, wf, nrm[n], nrm[kSeq + n]);  // xhat, BF16
                if constexpr (WT == MTP_W_FP8_E4M3) {
                  // f16 of xhat * 2^k (exact inside the f16 range)
                  const float xs = nrm[2 * kSeq + n];
                  auto f16x2 = [xs](uint32_t v) {
                    return f16x2_bits(__fmul_rn(bf16_lo(v), xs), __fmul_rn(bf16_hi(v), xs));
                  };
                  o = make_uint4(f16x2(o.x), f16x2(o.y), f16x2(o.z), f16x2(o.w));
                }
              }
              *reinterpret_cast<uint4*>(bt_base + sub * 2048 + swz(n, c)) = o;
            }
          }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bfull[slot]));
        if (++slot == kBStages) { slot = 0; ep ^= 1u; }
        if (u + 1 < nstages) fetch(u + 1);
      }
    } else {
      // ---------------------------------------------------------------- consumers
      named_barrier_sync(1, kPrologueThreads);  // pairs with the builders' wait for the factors
      const int g = lane >> 2, t4 = lane & 3;
      ArgBest best[NT][2];
#pragma unroll
      for (int jn = 0; jn < NT; ++jn) best[jn][0] = best[jn][1] = ArgBest{0.0f, -1};
      int aslot = 0, bslot = 0;
      uint32_t ap = 0, bp = 0;
      bool ok = true;
      for (int gt = t0; gt < t1 && ok; gt += kTileGroup) {
        const int ntile = (t1 - gt) < kTileGroup ? (t1 - gt) : kTileGroup;
        float acc[kTileGroup][NT][4];
#pragma unroll
        for (int j = 0; j < kTileGroup; ++j)
#pragma unroll
          for (int jn = 0; jn < NT; ++jn) acc[j][jn][0] = acc[j][jn][1] = acc[j][jn][2] = acc[j][jn][3] = 0.0f;
        // row scales of the FP8 head for this thread's rows, loaded ahead of the epilogue
        float scl[kTileGroup][2];
#pragma unroll
        for (int j = 0; j < kTileGroup; ++j) {
          scl[j][0] = scl[j][1] = 1.0f;
          if constexpr (WT == MTP_W_FP8_E4M3) {
            const int64_t r0 = static_cast<int64_t>(gt + j) * kTileRows + 16 * warp + g;
            if (j < ntile && r0 < V) scl[j][0] = __ldg(a.scale + r0);
            if (j < ntile && r0 + 8 < V) scl[j][1] = __ldg(a.scale + r0 + 8);
          }
        }
        for (int kp = 0; kp < KP && ok; ++kp) {
          const int nsub = KB - kp * kKS < kKS ? KB - kp * kKS : kKS;
          if (*reinterpret_cast<volatile int*>(&abort_flag) ||
              !__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&bfull[bslot]), bp, a.wait_ns))) {
            ok = false;
            break;
          }
          BFrags<WT, NT> bf[kKS];
#pragma unroll
          for (int sb = 0; sb < kKS; ++sb) bf[sb].load(smem_addr(bring + bslot * BSB + sb * BTB), lane);
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&bempty[bslot]));
          if (++bslot == kBStages) { bslot = 0; bp ^= 1u; }
#pragma unroll
          for (int j = 0; j < kTileGroup; ++j) {
            if (j < ntile && ok) {
              if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&afull[aslot]), ap, a.wait_ns))) {
                ok = false;
              } else {
#pragma unroll
                for (int sb = 0; sb < kKS; ++sb)
                  if (sb < nsub) bf[sb].mma(smem_addr(aring + aslot * kAStageBytes + sb * kATileBytes), acc[j], warp, lane);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&aempty[aslot]));
                if (++aslot == kAStages) { aslot = 0; ap ^= 1u; }
              }
            }
          }
        }
        if (!ok) break;
        // epilogue of the group: logits and per-sequence running argmax
#pragma unroll
        for (int j = 0; j < kTileGroup; ++j) {
          if (j < ntile) {
            const int64_t rbase = static_cast<int64_t>(gt + j) * kTileRows + 16 * warp + g;
#pragma unroll
            for (int jn = 0; jn < NT; ++jn) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int n = 8 * jn + 2 * t4 + (i & 1);
                const int64_t row = rbase + 8 * (i >> 1);
                if (n < B && row < V) {
                  float v = acc[j][jn][i];
                  if constexpr (WT == MTP_W_FP8_E4M3) v = __fmul_rn(__fmul_rn(v, nrm[3 * kSeq + n]), scl[j][i >> 1]);
                  if (a.logits != nullptr) a.logits[static_cast<int64_t>(n) * V + row] = v;
                  arg_update(best[jn][i & 1], v, static_cast<int32_t>(row));
                }
              }
            }
          }
        }
      }
      if (!ok && lane == 0) {
        store_status(a.status, MTP_ERR_TIMEOUT);
        atomicExch(&abort_flag, 1);
      }
      // combine lanes that hold the same sequences (same t4), then publish per warp
#pragma unroll
      for (int jn = 0; jn < NT; ++jn)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          ArgBest b = best[jn][hh];
#pragma unroll
          for (int m = 4; m < 32; m <<= 1) {
            const float v = __shfl_xor_sync(0xffffffffu, b.v, m);
            const int32_t i = __shfl_xor_sync(0xffffffffu, b.i, m);
            if (i >= 0) arg_update(b, v, i);
          }
          const int n = 8 * jn + 2 * t4 + hh;
          if (g == 0 && n < B) wbest[warp * kSeq + n] = b;
        }
    }
  }
  __syncthreads();
  pdl_wait_prior_grid();  // the workspace may still be read by the kernel before (no-op if done)
  tc_argmax_finish(B, wbest, a);
}

// ---------------------------------------------------------------------------- host side
template <int WT, int NT>
cudaError_t launch_tc(const SweepArgs& a, const CUtensorMap& tm, unsigned grid, size_t smem, cudaStream_t stream) {
  SweepArgs args = a;
  CUtensorMap tmc = tm;
  void* params[] = {&tmc, &args};
  return launch_pdl(reinterpret_cast<const void*>(sweep_tc_kernel<WT, NT>), dim3(grid), dim3(kTcThreads), smem,
                    stream, params);
}

}  // namespace

size_t sweep_tc_smem_bytes(int w_dtype) {
  const int bsb = (w_dtype == MTP_W_BF16) ? TcCfg<MTP_W_BF16>::kBStageBytes : TcCfg<MTP_W_FP8_E4M3>::kBStageBytes;
  const int nbs = (w_dtype == MTP_W_BF16) ? TcCfg<MTP_W_BF16>::kBStages : TcCfg<MTP_W_FP8_E4M3>::kBStages;
  return 1024 + static_cast<size_t>(kAStages) * kAStageBytes + static_cast<size_t>(nbs) * bsb +
         (2 * kAStages + 2 * nbs) * 8 + 4 * kSeq * 4 + kTcWarps * kSeq * sizeof(ArgBest) + 64;
}

cudaError_t launch_sweep_tc(const SweepArgs& a, cudaStream_t stream, bool* launched) {
  *launched = false;
  const int EB = (a.w_dtype == MTP_W_BF16) ? 2 : 1;
  if (a.B < 2 || a.B > kSeq) return cudaSuccess;
  if ((static_cast<int64_t>(a.H) * EB) % 16 != 0 || (a.H % 8) != 0) return cudaSuccess;
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  const size_t smem = sweep_tc_smem_bytes(a.w_dtype);
  if (smem > static_cast<size_t>(di.smem_optin)) return cudaSuccess;
  const TmapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaSuccess;
  CUtensorMap tm;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.H), static_cast<cuuint64_t>(a.V)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.H) * EB};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(a.w_dtype == MTP_W_BF16 ? 64 : 128),
                             static_cast<cuuint32_t>(kTileRows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult cr = enc(&tm, a.w_dtype == MTP_W_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                          2, const_cast<uint8_t*>(a.W), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return cudaSuccess;
  const int64_t T = (static_cast<int64_t>(a.V) + kTileRows - 1) / kTileRows;
  int64_t g = di.sm_count < T ? di.sm_count : T;
  if (g > kMaxGrid) g = kMaxGrid;
  const unsigned grid = static_cast<unsigned>(g < 1 ? 1 : g);
  *launched = true;
  {
    SweepArgs na = a;
    void* nparams[] = {&na};
    const void* nk = a.w_dtype == MTP_W_BF16 ? reinterpret_cast<const void*>(xnorm_parts_kernel<MTP_W_BF16>)
                                             : reinterpret_cast<const void*>(xnorm_parts_kernel<MTP_W_FP8_E4M3>);
    err = launch_pdl(nk, dim3(kNormParts, a.B), dim3(32), 0, stream, nparams);
    if (err != cudaSuccess) return err;
  }
  if (a.w_dtype == MTP_W_BF16)
    return a.B <= 8 ? launch_tc<MTP_W_BF16, 1>(a, tm, grid, smem, stream) : launch_tc<MTP_W_BF16, 2>(a, tm, grid, smem, stream);
  return a.B <= 8 ? launch_tc<MTP_W_FP8_E4M3, 1>(a, tm, grid, smem, stream)
                  : launch_tc<MTP_W_FP8_E4M3, 2>(a, tm, grid, smem, stream);
}

}  // namespace mtp
