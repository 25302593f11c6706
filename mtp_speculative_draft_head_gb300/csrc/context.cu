// Context-row input stage ("glm5next_mtp_head.rs", `rows_impl`: for every context row r the
// embedding row of tokens[r] and hidden row r go through enorm / hnorm, the concat and eh_proj --
// the input stage of `forward_one` per row; the source loops over rows on the host, here all R
// rows run at once).
//
// Kernels:
//  1. context_concat_rows_kernel (few rows: one CTA per row) or context_concat_warps_kernel
//     (many rows: one warp per vector) forms the concat rows [enorm(e_r) | hnorm(h_r)] (the same
//     correctly rounded BF16 values as the single-sequence kernels) in the workspace, plus a
//     flag per row for the token check.
//  2. context_gemm_kernel: x = concat . eh_proj^T, an R x H x 2H GEMM -- compute-bound once R
//     reaches a few hundred rows, so it runs on the fifth-generation tensor cores: 256 x 256
//     output tiles (two 128 x 256 FP32 accumulators in TMEM sharing each eh_proj tile), operands
//     streamed by 2-D TMA tensor loads (128-byte swizzle, the K-major layout the MMA reads
//     directly) into a 3-stage ring, one thread issuing tcgen05.mma (BF16 x BF16), one
//     warpgroup per accumulator moving it out of TMEM, rounding it to BF16 and storing x. FP32
//     accumulation is the source's precision for eh_proj. Whole waves of tiles run one CTA per
//     tile; the tiles of a last, partial wave are split along k into equal ranges, whose CTAs
//     store FP32 partial sums, which
//  3. context_reduce_kernel adds in k order and rounds to BF16 (deterministic).
// Warp roles of the GEMM: warp 0 lane 0 = TMA producer, warp 1 = TMEM allocation and (lane 0)
// MMA issue, warps 4..7 / 8..11 = epilogue of accumulator 0 / 1 (warp w reads TMEM lanes
// 32 (w % 4) ...).
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

// ------------------------------------------------------------------------------- concat
// Both forms compute what the single-sequence kernels compute: squares of BF16 values (exact in
// fp32) summed as double-floats, 1/rms = rsqrt(mean + eps) in fp64 split into two fp32 parts,
// and x * w * (1/rms) rounded once to BF16 from a double-float (bf16x8_scaled_rne), so every
// output is the correctly rounded BF16 value whatever the summation order.
//
// Few rows (latency-bound): one CTA of 512 threads per row, both vectors at once, a handful of
// 16-byte pieces per thread (the shared norm prologue).
#ifndef MTP_CTX_CAT
#define MTP_CTX_CAT 0  // concat kernel: 0 chosen by row count, 1 one CTA per row, 2 one warp per vector
#endif
constexpr int kCtxNormThreads = 512;

__global__ void __launch_bounds__(kCtxNormThreads) context_concat_rows_kernel(const ContextArgs a) {
  __shared__ float red[2 * (2 * kCtxNormThreads / 32 + 2)];
  __shared__ int ok_s;
  const int r = blockIdx.x;
  const int H = a.H;
  // The GEMM may launch at once, before this grid even waits for the kernel before it: its
  // producer streams eh_proj (which depends on nothing) and waits for this grid's completion
  // before it reads the concat. Launched this early, its CTAs take the SMs that the preceding
  // kernel's CTAs leave as they finish, and its weight stream fills the HBM time that the end of
  // that kernel leaves idle (a batched draft chain, after a sweep: 1.4 to 4 us a step, B = 2..16).
  // Every CTA of this grid has started by the time the GEMM launches, so the GEMM never holds
  // SMs this grid still needs.
  pdl_launch_dependents();
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
}

// Many rows (bandwidth-bound): one warp per normalised vector (vector 2r: enorm of the embedding
// row of tokens[r]; 2r + 1: hnorm of hidden row r), no block-level synchronisation, many vectors
// in flight per SM. Pass 1 reads x in batches of kCatBatch 16-byte pieces per lane (all in
// flight together) into four packed pairs of double-float sums; pass 2 reads x again (L1 / L2)
// with the norm weight, again a batch at a time.
constexpr int kCatWarps = 8;
constexpr int kCatBatch = 8;

__global__ void __launch_bounds__(kCatWarps * 32, 4) context_concat_warps_kernel(const ContextArgs a) {
  pdl_wait_prior_grid();  // tokens and target_hidden may come from the preceding kernel
  const int lane = threadIdx.x & 31;
  const int H = a.H, nv8 = a.H / 8;
  const int64_t nvec = 2 * static_cast<int64_t>(a.R);
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t vec = static_cast<int64_t>(blockIdx.x) * kCatWarps + (threadIdx.x >> 5); vec < nvec;
       vec += static_cast<int64_t>(gridDim.x) * kCatWarps) {
    const int r = static_cast<int>(vec >> 1), half = static_cast<int>(vec & 1);
    const uint16_t* x;
    const uint16_t* w;
    bool ok = true;
    if (half == 0) {
      const int32_t tok = a.tokens[r];
      ok = tok >= 0 && tok < a.V;
      if (lane == 0) {
        a.valid[r] = ok ? 1 : 0;
        if (!ok) store_status(a.status, MTP_ERR_TOKEN_RANGE);
      }
      x = a.embed + static_cast<int64_t>(ok ? tok : 0) * H;
      w = a.enorm_w;
    } else {
      x = a.hidden + static_cast<size_t>(r) * H;
      w = a.hnorm_w;
    }
    uint4* out = reinterpret_cast<uint4*>(a.concat + static_cast<size_t>(r) * 2 * H + static_cast<size_t>(half) * H);
    const uint4* xv = reinterpret_cast<const uint4*>(x);
    const uint4* wv = reinterpret_cast<const uint4*>(w);
    if (!ok) {  // the embedding table is not read for an out-of-range token
      for (int v = lane; v < nv8; v += 32) out[v] = z;
      continue;
    }
    // four packed pairs of double-float sums (f32x2: two TwoSums per instruction sequence);
    // each square of a BF16 value is exact in fp32
    DF2 acc[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) acc[t] = DF2{0ull, 0ull};
    for (int v0 = 0; v0 < nv8; v0 += 32 * kCatBatch) {
      uint4 q[kCatBatch];
#pragma unroll
      for (int i = 0; i < kCatBatch; ++i) {
        const int v = v0 + 32 * i + lane;
        q[i] = v < nv8 ? xv[v] : z;
      }
#pragma unroll
      for (int i = 0; i < kCatBatch; ++i) {
        const uint32_t u[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint64_t x2 = bf16x2_to_f2(u[t]);
          df2_add(acc[t], f2_mul(x2, x2));
        }
      }
    }
    DF tot = df_add(df_add(df_add(df2_x(acc[0]), df2_y(acc[0])), df_add(df2_x(acc[1]), df2_y(acc[1]))),
                    df_add(df_add(df2_x(acc[2]), df2_y(acc[2])), df_add(df2_x(acc[3]), df2_y(acc[3]))));
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) tot = df_add(tot, shfl_xor_df(tot, m));
    const double ms = (static_cast<double>(tot.hi) + static_cast<double>(tot.lo)) * a.inv_h;
    const double rinv = rsqrt(ms + static_cast<double>(a.eps));
    const float rh = static_cast<float>(rinv);
    const float rl = static_cast<float>(rinv - static_cast<double>(rh));
    constexpr int kB2 = kCatBatch / 2;
    for (int v0 = 0; v0 < nv8; v0 += 32 * kB2) {
      uint4 xq[kB2], wq[kB2];
#pragma unroll
      for (int i = 0; i < kB2; ++i) {
        const int v = v0 + 32 * i + lane;
        xq[i] = v < nv8 ? xv[v] : z;
        wq[i] = v < nv8 ? wv[v] : z;
      }
#pragma unroll
      for (int i = 0; i < kB2; ++i) {
        const int v = v0 + 32 * i + lane;
        if (v < nv8) {
          const uint32_t xu[4] = {xq[i].x, xq[i].y, xq[i].z, xq[i].w};
          const uint4 w4 = wq[i];
          const float wf[8] = {bf16_lo(w4.x), bf16_hi(w4.x), bf16_lo(w4.y), bf16_hi(w4.y),
                               bf16_lo(w4.z), bf16_hi(w4.z), bf16_lo(w4.w), bf16_hi(w4.w)};
          out[v] = bf16x8_scaled_rne(xu, wf, rh, rl);
        }
      }
    }
  }
  pdl_launch_dependents();
}

// ------------------------------------------------------------------------------- GEMM
#ifndef MTP_CTX_TILES
#define MTP_CTX_TILES 0  // 0: tile height chosen per shape (make_sched); 1 / 2: 128- / 256-row tiles only
#endif
#ifndef MTP_CTX_SPLITS
#define MTP_CTX_SPLITS 0  // 0: schedule chosen per shape (make_sched); 1: whole tiles only; 2: always split the last wave
#endif
constexpr int kGN = 256;                  // output columns (x features) per tile
constexpr int kGK = 64;                   // k elements per stage (one 128-byte swizzle atom)
constexpr int kGBBytes = kGN * kGK * 2;   // 32 KB of eh_proj per stage
#ifndef MTP_CTX_L2_AHEAD
#define MTP_CTX_L2_AHEAD 8
#endif
constexpr int kCtxL2Ahead = MTP_CTX_L2_AHEAD;  // eh_proj tiles prefetched into L2 past the ring at the start

// Tile of HALVES 128 x 256 FP32 accumulators (TMEM) over HALVES * 128 context rows.
template <int HALVES>
struct Tile {
  static constexpr int kHalves = HALVES;
  static constexpr int kM = 128 * HALVES;                  // output rows (context rows) per tile
  static constexpr int kStages = HALVES == 2 ? 3 : 4;      // ring depth that fits shared memory
  static constexpr int kABytes = kM * kGK * 2;             // 16 KB per 128-row half
  static constexpr int kStageBytes = kABytes + kGBBytes;
  static constexpr int kThreads = 128 + 128 * HALVES;      // 4 role warps + one epilogue warpgroup per half
  static constexpr uint32_t kTmemCols = kGN * HALVES;      // 128 lanes x 256 columns per accumulator
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(kStages) * kStageBytes + (2 * kStages + 1) * 8 + 16;
  static_assert(kTmemCols <= 512, "TMEM holds 512 columns");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// Tile height: the kernel is limited by the operand bytes in flight per SM (a ring of a few
// stages against the L2 / HBM latency), so the tile that does the most MMA work per byte wins
// when there are enough tiles: two 128 x 256 accumulators fed by one 256-row A tile and one
// shared 256-row eh_proj tile do 128 flops per staged byte, against 85 for a single 128 x 256
// tile. The single-accumulator tile has a deeper ring (4 stages) and twice as many tiles, which
// wins for few rows (the eh_proj stream is the bound) and where it fills the SMs better.
//
// Work split. Tiles t = 0 .. T-1 run with the row tile fastest, so the CTAs of a wave share
// eh_proj tiles. The first n_dp tiles are whole waves of CTAs, one tile each, writing x in BF16.
// The n_rem tiles after them (a last, partial wave) are split along k into `splits` equal
// ranges: CTA n_dp + s * n_rem + r takes k range s of tile n_dp + r, so the CTAs of one range
// start together and the row tiles of an eh_proj tile read it at the same time (one HBM read,
// the rest from L2), and no SM idles for a whole tile's time. Those CTAs write FP32 partial sums
// into slot r * splits + s, and context_reduce_kernel adds each tile's partials in k order.
struct CtxSched {
  int halves;      // tile height: 128 * halves rows
  int tile_m;      // 128 * halves
  int mt;          // row tiles
  int nkb;         // k-blocks per tile
  int n_dp;        // tiles done whole, one CTA each: CTAs 0 .. n_dp-1
  int n_rem;       // tiles n_dp .. n_dp+n_rem-1, split along k
  int splits;      // k ranges per split tile (1: the remaining tiles are whole too)
  int slot_rows;   // rows of a partial slot: min(R, tile_m)
};

template <int HALVES>
__global__ void __launch_bounds__(Tile<HALVES>::kThreads, 1)
    context_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                        const ContextArgs a, const CtxSched c) {
  using TC = Tile<HALVES>;
  constexpr int kGHalves = TC::kHalves, kGM = TC::kM, kGStages = TC::kStages, kGABytes = TC::kABytes;
  constexpr int kGStageBytes = TC::kStageBytes;
  constexpr uint32_t kTmemCols = TC::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kGStages * kGStageBytes);
  uint64_t* empty = full + kGStages;
  uint64_t* acc_full = empty + kGStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this CTA's tile and k range
  int t, kb0, nkb, slot = -1;
  if (static_cast<int>(blockIdx.x) < c.n_dp || c.splits == 1) {
    t = blockIdx.x;
    kb0 = 0;
    nkb = c.nkb;
  } else {
    const int i = static_cast<int>(blockIdx.x) - c.n_dp;
    const int sp = i / c.n_rem, r = i % c.n_rem;
    t = c.n_dp + r;
    kb0 = sp * c.nkb / c.splits;
    nkb = (sp + 1) * c.nkb / c.splits - kb0;
    slot = r * c.splits + sp;
  }
  const int m0 = (t % c.mt) * kGM, n0 = (t / c.mt) * kGN;
  // 128-row halves of this tile that hold context rows (the rest of the A box is zero fill)
  const int halves = (a.R - m0) >= kGM ? kGHalves : (a.R - m0 + 127) / 128;

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
      const uint64_t pol_b = l2_evict_first_policy();
      uint64_t pol_a;
      asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_a));
      // eh_proj does not depend on the preceding kernel (the concat): the eh_proj half of the
      // first stages is in flight, and the next kCtxL2Ahead eh_proj tiles are on their way to L2,
      // before the wait for it. Each stage barrier expects both halves, so a stage completes once
      // its concat half, issued after the wait, has landed too.
      const int pre = nkb < kGStages ? nkb : kGStages;
      for (int kb = 0; kb < pre; ++kb) {
        const uint32_t bar = smem_addr(&full[kb]);
        mbar_arrive_expect_tx(bar, kGStageBytes);
        tma_load_2d(smem_addr(smem + kb * kGStageBytes + kGABytes), &tm_b, (kb0 + kb) * kGK, n0, bar, pol_b);
      }
      for (int kb = pre; kb < nkb && kb < pre + kCtxL2Ahead; ++kb) tma_prefetch_l2_2d(&tm_b, (kb0 + kb) * kGK, n0);
      pdl_wait_prior_grid();  // the concat comes from the preceding kernel
      for (int kb = 0; kb < pre; ++kb)
        tma_load_2d(smem_addr(smem + kb * kGStageBytes), &tm_a, (kb0 + kb) * kGK, m0, smem_addr(&full[kb]), pol_a);
      int issued = pre;
      for (int kb = pre; kb < nkb; ++kb) {
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
        tma_load_2d(smem_addr(st), &tm_a, (kb0 + kb) * kGK, m0, bar, pol_a);
        tma_load_2d(smem_addr(st + kGABytes), &tm_b, (kb0 + kb) * kGK, n0, bar, pol_b);
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
      constexpr uint32_t idesc = umma_idesc_bf16(128, kGN);
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
        const uint64_t db = umma_desc_sw128(sa + kGABytes);
#pragma unroll
        for (int k = 0; k < kGK / 16; ++k) {  // 16 elements = 32 bytes along the swizzle row
          const uint64_t koff = static_cast<uint64_t>((32 * k) >> 4);
          const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
#pragma unroll
          for (int hf = 0; hf < kGHalves; ++hf)  // half hf: A rows 128 hf.., accumulator columns 256 hf..
            if (hf < halves)
              umma_bf16(tmem + static_cast<uint32_t>(hf * kGN), umma_desc_sw128(sa + hf * 128 * 128) + koff,
                        db + koff, idesc, acc);
        }
        umma_commit(smem_addr(&empty[s]));  // the stage is free once these MMAs have read it
      }
      // always: the epilogue (and the TMEM release) wait for every issued MMA
      umma_commit(smem_addr(acc_full));
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int hf = (warp - 4) >> 2;  // accumulator half
    const int q = warp & 3;          // TMEM lanes 32 q .. 32 q + 31 (a warp reaches lanes 32 (warp % 4) ..)
    const bool done = mbar_wait_bounded(smem_addr(acc_full), 0);
    tmem_fence_after_sync();
    if (!done) {
      if (lane == 0) store_status(a.status, MTP_ERR_TIMEOUT);
    } else if (hf < halves && !*reinterpret_cast<volatile int*>(&abort_flag)) {
      const int lrow = 128 * hf + 32 * q + lane;  // row within the tile
      const int row = m0 + lrow;
      const bool row_ok = row < a.R;
      const bool valid = row_ok && a.valid[row] != 0;
      float* part = slot < 0 ? nullptr : a.partial + (static_cast<size_t>(slot) * c.slot_rows + lrow) * kGN;
#pragma unroll 1
      for (int c0 = 0; c0 < kGN; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(hf * kGN + c0), v);
        // H is a multiple of 32, so a 32-column slice is inside x or outside it as a whole
        if (!row_ok || n0 + c0 >= a.H) continue;
        if (part != nullptr) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            reinterpret_cast<uint4*>(part + c0)[e] = make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
        } else {
          uint16_t* dst = a.x + static_cast<size_t>(row) * a.H + n0 + c0;
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const uint32_t lo = valid ? bf16_bits_rn(__uint_as_float(v[2 * e])) : 0u;
            const uint32_t hi = valid ? bf16_bits_rn(__uint_as_float(v[2 * e + 1])) : 0u;
            w[e] = lo | (hi << 16);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e)
            reinterpret_cast<uint4*>(dst)[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
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

// x = bf16( sum of a split tile's partial slots in k order ), zeros for rows whose token is out
// of range. One thread per 8 outputs.
__global__ void __launch_bounds__(256) context_reduce_kernel(const ContextArgs a, const CtxSched c) {
  pdl_wait_prior_grid();  // the partials come from the GEMM
  const int64_t per_tile = static_cast<int64_t>(c.slot_rows) * (kGN / 8);
  const int64_t total = per_tile * c.n_rem;
  const size_t slot_floats = static_cast<size_t>(c.slot_rows) * kGN;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(idx / per_tile);
    const int lrow = static_cast<int>((idx % per_tile) / (kGN / 8));
    const int col8 = static_cast<int>(idx % (kGN / 8));
    const int t = c.n_dp + r;
    const int row = (t % c.mt) * c.tile_m + lrow;
    const int col = (t / c.mt) * kGN + 8 * col8;
    if (row >= a.R || col >= a.H) continue;
    const float* p = a.partial + static_cast<size_t>(r) * c.splits * slot_floats + static_cast<size_t>(lrow) * kGN +
                     8 * col8;
    float4 lo = *reinterpret_cast<const float4*>(p), hi = *reinterpret_cast<const float4*>(p + 4);
    for (int sp = 1; sp < c.splits; ++sp) {
      const float4 l = *reinterpret_cast<const float4*>(p + sp * slot_floats);
      const float4 h = *reinterpret_cast<const float4*>(p + sp * slot_floats + 4);
      lo.x += l.x; lo.y += l.y; lo.z += l.z; lo.w += l.w;
      hi.x += h.x; hi.y += h.y; hi.z += h.z; hi.w += h.w;
    }
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (a.valid[row] != 0)
      o = make_uint4(bf16_bits_rn(lo.x) | (bf16_bits_rn(lo.y) << 16), bf16_bits_rn(lo.z) | (bf16_bits_rn(lo.w) << 16),
                     bf16_bits_rn(hi.x) | (bf16_bits_rn(hi.y) << 16), bf16_bits_rn(hi.z) | (bf16_bits_rn(hi.w) << 16));
    *reinterpret_cast<uint4*>(a.x + static_cast<size_t>(row) * a.H + col) = o;
  }
  pdl_launch_dependents();
}

// Workspace: the concat [R, 2H] BF16, the row flags [R] int32, then kMaxSlots partial slots of
// min(R, 256) x 256 FP32 (the split tiles times their k ranges never exceed it).
constexpr int kMaxSlots = 320;
constexpr int kMaxSplits = 16;

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// The work split: a small cost model in microseconds picks the tile height and whether the tiles
// of a last, partial wave are split along k (and how many ways). A k-block takes kb_us on the
// tensor cores (measured: ~0.76 us for a full 256-row tile, ~0.43 us for a 128-row tile or a
// 256-row tile with one half in use), a CTA's start-up and epilogue kCtaUs; eh_proj and the
// concat must come from HBM at least once (kHbmBytesPerUs); splitting adds the partials' write
// and read-back and one more launch. The model only picks among correct schedules.
CtxSched make_sched_for(int halves, int R, int H, int sm_count, double* est_us) {
  // kSmBytesPerUs: the eh_proj bytes one CTA streams per us, about the HBM rate over all SMs (at
  // R = 17, 96 CTAs of 48 k-blocks each took 25.5 us: 5.8 TB/s, 60 GB/s per SM); a wave of fewer
  // CTAs than the HBM rate needs cannot reach the HBM roofline.
  constexpr double kCtaUs = 2.5, kHbmBytesPerUs = 6.5e6, kLaunchUs = 2.0, kSmBytesPerUs = 5.0e4;
  CtxSched c{};
  c.halves = halves;
  c.tile_m = 128 * halves;
  c.mt = (R + c.tile_m - 1) / c.tile_m;
  c.nkb = 2 * H / kGK;
  c.slot_rows = R < c.tile_m ? R : c.tile_m;
  const int T = c.mt * ((H + kGN - 1) / kGN);
  const int G = sm_count;
  const double kb_us = (halves == 2 && R > 128) ? 0.76 : 0.43;
  // HBM floor of a wave of `ctas` CTAs over `tiles` tiles: the row tiles of one eh_proj column
  // tile (kGN rows x 2H) read it from HBM once, the rest from L2, so a tile stands for 1 / mt of
  // an eh_proj tile; the concat (all R rows) is read once too (cat_us)
  const double tile_bytes = static_cast<double>(kGN) * 2 * H * 2 / c.mt;
  auto hbm_floor = [&](double tiles, int64_t ctas) {
    const double rate = ctas * kSmBytesPerUs < kHbmBytesPerUs ? ctas * kSmBytesPerUs : kHbmBytesPerUs;
    return tiles * tile_bytes / rate;
  };
  const double cat_us = 2.0 * R * 2 * H / kHbmBytesPerUs;
  const double tile_us = c.nkb * kb_us + kCtaUs;
  auto at_least = [](double us, double floor) { return us > floor ? us : floor; };
  c.n_dp = T;
  c.n_rem = 0;
  c.splits = 1;
  double best = at_least(static_cast<double>((T + G - 1) / G) * tile_us, hbm_floor(T, T < G ? T : G) + cat_us);
  const int n_dp = (T / G) * G, n_rem = T - n_dp;
  for (int sp = 2; MTP_CTX_SPLITS != 1 && n_rem > 0 && sp <= kMaxSplits && sp <= c.nkb && n_rem * sp <= kMaxSlots;
       ++sp) {
    const int64_t rem_ctas = static_cast<int64_t>(n_rem) * sp;
    const int64_t waves = (rem_ctas + G - 1) / G;
    const double part_bytes = static_cast<double>(n_rem) * sp * c.slot_rows * kGN * 4;
    const double floor = hbm_floor(n_dp, G) + hbm_floor(n_rem, rem_ctas < G ? rem_ctas : G) + cat_us;
    const double us = at_least(static_cast<double>(n_dp / G) * tile_us +
                                   static_cast<double>(waves) * (((c.nkb + sp - 1) / sp) * kb_us + kCtaUs),
                               floor) +
                      2.0 * part_bytes / kHbmBytesPerUs + kLaunchUs;
    if (us < best || (MTP_CTX_SPLITS > 1 && c.splits == 1)) {
      best = us;
      c.n_dp = n_dp;
      c.n_rem = n_rem;
      c.splits = sp;
    }
  }
  *est_us = best;
  return c;
}

CtxSched make_sched(int R, int H, int sm_count) {
  double e1 = 0.0, e2 = 0.0;
  const CtxSched c1 = make_sched_for(1, R, H, sm_count, &e1);
  const CtxSched c2 = make_sched_for(2, R, H, sm_count, &e2);
  if (MTP_CTX_TILES == 1) return c1;
  if (MTP_CTX_TILES == 2) return c2;
  return e2 < e1 ? c2 : c1;
}

}  // namespace

size_t context_workspace_bytes(int R, int H) {
  return round256(static_cast<size_t>(R) * 2 * H * 2) + round256(static_cast<size_t>(R) * 4) +
         static_cast<size_t>(kMaxSlots) * (R < 256 ? R : 256) * kGN * 4;
}

void bind_context_workspace(ContextArgs* a, void* ws) {
  uint8_t* p = static_cast<uint8_t*>(ws);
  a->concat = reinterpret_cast<uint16_t*>(p);
  p += round256(static_cast<size_t>(a->R) * 2 * a->H * 2);
  a->valid = reinterpret_cast<int32_t*>(p);
  p += round256(static_cast<size_t>(a->R) * 4);
  a->partial = reinterpret_cast<float*>(p);
}

cudaError_t launch_context_concat(const ContextArgs& in, cudaStream_t stream) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  ContextArgs a = in;
  void* params[] = {&a};
  // one warp per vector once there are enough vectors (measured: from about a thousand rows)
  const bool warps = MTP_CTX_CAT == 2 || (MTP_CTX_CAT == 0 && 2 * static_cast<int64_t>(a.R) >= 2LL * kCatWarps * di.sm_count);
  if (warps) {
    int64_t blocks = (2 * static_cast<int64_t>(a.R) + kCatWarps - 1) / kCatWarps;
    if (blocks > 4 * di.sm_count) blocks = 4 * di.sm_count;
    return launch_pdl(reinterpret_cast<const void*>(context_concat_warps_kernel), dim3(static_cast<unsigned>(blocks)),
                      dim3(kCatWarps * 32), 0, stream, params);
  }
  return launch_pdl(reinterpret_cast<const void*>(context_concat_rows_kernel), dim3(static_cast<unsigned>(a.R)),
                    dim3(kCtxNormThreads), 0, stream, params);
}

cudaError_t launch_context_rows(const ContextArgs& in, cudaStream_t stream) {
  DeviceInfo di;
  cudaError_t err = device_info(&di);
  if (err != cudaSuccess) return err;
  if (in.H % 32 != 0) return cudaErrorNotSupported;
  const TmapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // one CTA per whole tile (row tiles fastest, so a wave shares eh_proj tiles), then the k ranges
  // of the split tiles (range index slowest)
  CtxSched c = make_sched(in.R, in.H, di.sm_count);
  const size_t smem = c.halves == 2 ? Tile<2>::kSmem : Tile<1>::kSmem;
  if (smem > static_cast<size_t>(di.smem_optin)) return cudaErrorNotSupported;
  ContextArgs a = in;
  const int K = 2 * a.H;
  CUtensorMap ta, tb;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(a.R)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {kGK, static_cast<cuuint32_t>(c.tile_m)};
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
  err = launch_context_concat(a, stream);
  if (err != cudaSuccess) return err;
  {
    CUtensorMap tac = ta, tbc = tb;
    void* params[] = {&tac, &tbc, &a, &c};
    const void* kern = c.halves == 2 ? reinterpret_cast<const void*>(context_gemm_kernel<2>)
                                     : reinterpret_cast<const void*>(context_gemm_kernel<1>);
    const int threads = c.halves == 2 ? Tile<2>::kThreads : Tile<1>::kThreads;
    err = launch_pdl(kern, dim3(static_cast<unsigned>(c.n_dp + c.n_rem * c.splits)), dim3(threads), smem, stream,
                     params);
    if (err != cudaSuccess || c.splits == 1) return err;
  }
  const int64_t items = static_cast<int64_t>(c.n_rem) * c.slot_rows * (kGN / 8);
  int64_t blocks = (items + 255) / 256;
  if (blocks > 4 * di.sm_count) blocks = 4 * di.sm_count;
  void* params[] = {&a, &c};
  return launch_pdl(reinterpret_cast<const void*>(context_reduce_kernel), dim3(static_cast<unsigned>(blocks)),
                    dim3(256), 0, stream, params);
}

}  // namespace mtp
