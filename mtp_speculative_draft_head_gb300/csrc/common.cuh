// Device building blocks shared by the MTP-head kernels (sm_103a).
//
//  * PTX wrappers: mbarrier, 1-D bulk async copy (TMA engine, global -> shared), L2 eviction
//    policy, async-proxy fence, programmatic dependent launch, global timer.
//  * Exact-rounding numerics: TwoSum, double-float accumulation, BF16 round-to-nearest-even
//    of a double-float value, the E4M3 bit-placement decode.
//  * Packed f32x2 arithmetic and packed double-float accumulation.
//  * The RMSNorm prologue (rms_norm_vanilla, x * w / rms) for several vectors, into shared memory.
//  * The (max, lowest index) argmax combine.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mtp_head.h"
#include "pick.h"

namespace mtp {

constexpr int kMaxB = 16;        // sequences per sweep
constexpr int kMaxGrid = 1024;   // CTAs per launch
// Output-stage workspace (kWsBytes, whatever B): the grid's finished-CTA counter at byte 0, the
// next dynamically claimed row (B = 1) at byte 64, from byte 128 each sequence's running pick
// (uint64 [kMaxB], below), and from byte 256 the batched sweep's norm parts: float4 {sum of
// squares hi, lo, max |x w|, 0} for kNormParts slices of each of up to kMaxB rows of x.
constexpr int kRowCounterOffset = 64;
constexpr int kWsPickOffset = 128;
constexpr int kNormParts = 8;
constexpr int kWsNormOffset = 256;
constexpr int kWsBytes = kWsNormOffset + kMaxB * kNormParts * 16;  // 2304
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // give up a wait after 2 s

// ------------------------------------------------------------------------------------------
// PTX wrappers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of an mbarrier, giving up after limit_ns (kWaitLimitNs unless the
// launch carries another limit for its stage waits). Returns false on timeout; the caller
// records MTP_ERR_TIMEOUT and stops. A limit of 0 gives up at once without looking at the
// barrier (the error path on demand). Waits for the kernel's own copies to land before it
// exits always take the default limit.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// L2 policy for data read exactly once per pass (weights far larger than L2).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D bulk copy global -> shared through the TMA engine, completing `bytes` transaction bytes
// on mbarrier `bar`. Requires 16-byte aligned addresses and a size that is a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// 2-D tensor tile global -> shared through the TMA engine (tensor map in kernel parameter space),
// completing on mbarrier `bar`. x (innermost coordinate) must start on a 16-byte boundary.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t bar,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}
// Prefetch a 2-D tensor tile into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void* tmap, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y)
               : "memory");
}
// Prefetch `bytes` contiguous bytes into L2 only (a hint: no completion to wait for). Address
// and size must be multiples of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Barrier over a subset of the block's warps (hardware named barrier `id`, `nthreads` threads).
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid (no-op when the launch did not
// ask for it), and allow the next grid to be scheduled.
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void store_status(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// ------------------------------------------------------------------------------------------
// Numerics
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }

// s + e == a + b exactly (Knuth's TwoSum; no ordering requirement on |a|, |b|).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// Double-float value hi + lo.
struct DF {
  float hi, lo;
};

__device__ __forceinline__ void df_add(DF& acc, float g) {
  float s, e;
  two_sum(acc.hi, g, s, e);
  acc.hi = s;
  acc.lo = __fadd_rn(acc.lo, e);
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  DF r;
  two_sum(s, e, r.hi, r.lo);
  return r;
}

__device__ __forceinline__ DF shfl_xor_df(DF v, int m) {
  DF r;
  r.hi = __shfl_xor_sync(0xffffffffu, v.hi, m);
  r.lo = __shfl_xor_sync(0xffffffffu, v.lo, m);
  return r;
}

// Round the exact value hi + lo to the nearest BF16 (ties to even). After renormalising,
// hi holds the value rounded to fp32 and lo the exact remainder (|lo| <= half an fp32 ulp), so
// only a hi that sits exactly on a BF16 midpoint needs lo to decide.
__device__ __forceinline__ uint16_t bf16_rne_df(float hi, float lo) {
  float s, e;
  two_sum(hi, lo, s, e);
  const uint32_t u = __float_as_uint(s);
  if ((u & 0x7F800000u) == 0x7F800000u) {  // inf or NaN
    if (u & 0x007FFFFFu) return static_cast<uint16_t>(((u >> 16) & 0x8000u) | 0x7FC0u);
    return static_cast<uint16_t>(u >> 16);
  }
  const uint32_t rem = u & 0xFFFFu;
  const uint32_t base = u >> 16;
  bool up;
  if (rem > 0x8000u) {
    up = true;
  } else if (rem < 0x8000u) {
    up = false;
  } else if (e == 0.0f) {
    up = (base & 1u) != 0u;
  } else {
    up = ((__float_as_uint(e) ^ u) & 0x80000000u) == 0u;  // same sign: larger magnitude
  }
  return static_cast<uint16_t>(base + (up ? 1u : 0u));
}

// BF16 (round to nearest even) of the double-float p * (rh + rl) as bf16_rne_df(yh, yl) with
// yh = fl(p * rh), yl = fl(p * rl + (p * rh - yh)) -- bit for bit, but cheaper: |yl| stays below
// 1.5 fp32 ulps of yh (|p * rh - yh| <= 0.5 ulp, |p * rl| < 1 ulp since |rl| <= ulp(rh) / 2), so
// the BF16 rounding of yh + yl can differ from that of yh alone only when yh lies within a few
// fp32 ulps of a BF16 midpoint (low 16 bits 0x7FFE..0x8002); those, inf / NaN, and a
// subnormal rh (where |rl| <= ulp(rh) / 2 no longer bounds p * rl by an ulp of yh) take the
// exact path.
// (The exact path is out of line: inlined into every element it doubled the cost of the
// common one.)
static __device__ __noinline__ uint32_t bf16_scaled_rne_exact(float p, float rh, float rl) {
  const float yh = __fmul_rn(p, rh);
  const float yl = __fmaf_rn(p, rl, __fmaf_rn(p, rh, -yh));
  return bf16_rne_df(yh, yl);
}
__device__ __forceinline__ uint32_t bf16_scaled_rne(float p, float rh, float rl) {
  const float yh = __fmul_rn(p, rh);
  const uint32_t u = __float_as_uint(yh);
  if (((u & 0xFFFFu) - 0x7FFEu) <= 4u || (u & 0x7F800000u) == 0x7F800000u || !(rh >= 1.17549435e-38f))
    return bf16_scaled_rne_exact(p, rh, rl);
  unsigned short h;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(yh));
  return h;
}

// Eight values at once: BF16 of x_i * w_i * (rh + rl) for the BF16 pairs xu[t] (elements 2t,
// 2t+1) and fp32 weights wf[i], packed in pairs -- the same bits as bf16_scaled_rne per element.
// The common path is straight-line (one packed conversion per pair); a cell with any element
// near a midpoint, inf / NaN, or a subnormal rh is redone on the exact path as a whole.
__device__ __forceinline__ uint4 bf16x8_scaled_rne(const uint32_t (&xu)[4], const float (&wf)[8], float rh,
                                                   float rl) {
  float p[8], y[8];
  uint32_t flag = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    p[i] = __fmul_rn((i & 1) ? bf16_hi(xu[i >> 1]) : bf16_lo(xu[i >> 1]), wf[i]);  // exact
    y[i] = __fmul_rn(p[i], rh);
    const uint32_t u = __float_as_uint(y[i]);
    flag |= static_cast<uint32_t>(((u - 0x7FFEu) & 0xFFFFu) <= 4u) | static_cast<uint32_t>((u & 0x7F800000u) == 0x7F800000u);
  }
  uint32_t o[4];
  if (flag == 0u && rh >= 1.17549435e-38f) {
#pragma unroll
    for (int t = 0; t < 4; ++t) asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[t]) : "f"(y[2 * t + 1]), "f"(y[2 * t]));
  } else {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float h0 = y[2 * t], h1 = y[2 * t + 1];
      const float l0 = __fmaf_rn(p[2 * t], rl, __fmaf_rn(p[2 * t], rh, -h0));
      const float l1 = __fmaf_rn(p[2 * t + 1], rl, __fmaf_rn(p[2 * t + 1], rh, -h1));
      o[t] = static_cast<uint32_t>(bf16_rne_df(h0, l0)) | (static_cast<uint32_t>(bf16_rne_df(h1, l1)) << 16);
    }
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// E4M3 byte i (0..3) of a 32-bit word -> fp32 holding value * 2^-120, exactly.
// The byte S.EEEE.MMM is placed as fp32 sign S, exponent field 0000EEEE and mantissa MMM:
// exponent field E gives 2^(E-127) * 1.MMM = 2^-120 * 2^(E-7) * 1.MMM; field 0 gives the fp32
// subnormal 2^-126 * MMM/8 = 2^-120 * 2^-6 * MMM/8 -- the E4M3 subnormal scaled the same way.
// (The NaN code S.1111.111 is never produced by the quantiser and decodes to a finite value.)
template <int I>
__device__ __forceinline__ float e4m3_byte_scaled(uint32_t w) {
  const int32_t t = static_cast<int32_t>(w << (24 - 8 * I)) >> 4;  // arithmetic shift
  return __uint_as_float(static_cast<uint32_t>(t) & 0x87F00000u);
}
constexpr float kE4m3Unscale = 1.329227995784915872903807060280344576e36f;  // 2^120

// ------------------------------------------------------------------------------------------
// Argmax: (value, index) pairs; larger value wins, equal values -> lower index, NaN never wins,
// index -1 marks "nothing yet".
// ------------------------------------------------------------------------------------------
struct ArgBest {
  float v;
  int32_t i;
};

__device__ __forceinline__ bool arg_beats(float v, int32_t i, const ArgBest& b) {
  if (v != v) return false;
  if (b.i < 0) return i >= 0;
  return v > b.v || (v == b.v && i < b.i);
}

__device__ __forceinline__ void arg_update(ArgBest& b, float v, int32_t i) {
  if (arg_beats(v, i, b)) {
    b.v = v;
    b.i = i;
  }
}

// The grid argmax across CTAs. Each CTA folds its best (value, row) of sequence b into a
// running maximum in the workspace by one 64-bit atomic max of the pick's exchange key (pick.h:
// its order is the argmax order, larger value first, then lower index; -0 counts as +0, and NaN
// never gets a key), stored with the top bit flipped so that 0 -- a zero-filled workspace -- is
// "no candidate yet". The last CTA to finish reads the B keys back (one load each), writes the
// drafts (and, for a vocabulary shard, the keys themselves), and puts the words back to 0 for
// the next launch. The maximum does not depend on the order of the atomics. (Before: each CTA
// wrote its partial, and the last CTA loaded and combined all of them, ncta x B partials: ~2.7
// to 4 us at B = 16 over 152 CTAs. The atomics took 0.6 to 3 us off every sweep, B = 1 to 16.)
__device__ __forceinline__ void pick_publish(uint8_t* ws, int b, float v, int32_t row, int32_t index_base) {
  if (row < 0) return;
  const uint64_t k = static_cast<uint64_t>(pick_key(v, row + index_base)) ^ 0x8000000000000000ull;
  atomicMax(reinterpret_cast<unsigned long long*>(ws + kWsPickOffset) + b, static_cast<unsigned long long>(k));
}

// Last CTA: the pick of sequence b into draft[b] (a global index, -1 if no row had a number)
// and pick[b] (may be null), and the running word back to 0.
__device__ __forceinline__ void pick_finish(uint8_t* ws, int b, int32_t* draft, int64_t* pick) {
  unsigned long long* kp = reinterpret_cast<unsigned long long*>(ws + kWsPickOffset) + b;
  const int64_t key = static_cast<int64_t>(static_cast<uint64_t>(__ldcg(kp)) ^ 0x8000000000000000ull);
  if (draft != nullptr) draft[b] = pick_index(key);
  if (pick != nullptr) pick[b] = key;
  *kp = 0ull;
}

// ------------------------------------------------------------------------------------------
// Packed fp32 pairs (sm_100+ f32x2 instructions): two IEEE round-to-nearest operations per
// instruction, lane-wise identical to the scalar ones.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
// (the first element of a packed pair is its low 32 bits)
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// BF16 pair (low half first) -> {f32(low), f32(high)}
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t u) {
  return f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// Two independent double-floats, packed: (hi.x, lo.x) and (hi.y, lo.y).
struct DF2 {
  uint64_t hi, lo;
};
// TwoSum of each lane's (hi, p), the error added to lo.
__device__ __forceinline__ void df2_add(DF2& a, uint64_t p) {
  const uint64_t s = f2_add(a.hi, p);
  const uint64_t bp = f2_sub(s, a.hi);
  const uint64_t e = f2_add(f2_sub(a.hi, f2_sub(s, bp)), f2_sub(p, bp));
  a.hi = s;
  a.lo = f2_add(a.lo, e);
}
__device__ __forceinline__ DF df2_x(const DF2& a) { return DF{f2_lo(a.hi), f2_lo(a.lo)}; }
__device__ __forceinline__ DF df2_y(const DF2& a) { return DF{f2_hi(a.hi), f2_hi(a.lo)}; }

// ------------------------------------------------------------------------------------------
// rms_norm_vanilla prologue for several vectors at once:
//   out_j = bf16( x_j * w_j / sqrt(mean(x_j^2) + eps) ), written into shared memory at layout(k).
// The sums of squares are double-floats (each square of a BF16 value is exact in fp32), 1/rms is
// formed in fp64 and split into two fp32 parts, and x*w (exact in fp32) times 1/rms is rounded
// once to BF16 from a double-float -- so each output is the correctly rounded BF16 of the fp64
// expression unless that lies within ~2^-40 relative of a rounding midpoint (1/rms is fp64 rsqrt,
// within an ulp or two of the correctly rounded fp64 value).
// One pass over the inputs, one block reduction for all vectors. All NT threads of the block
// call it; `red` holds >= njobs * (2 * NT / 32 + 2) floats. A job with valid == false writes
// zeros without reading x.
// ------------------------------------------------------------------------------------------
struct NormJob {
  const uint16_t* x;
  const uint16_t* w;
  uint16_t* out;
  bool valid;
};

struct NoOp {
  __device__ __forceinline__ void operator()() const {}
};

template <int NT, class Layout, class JobFn, class AfterLoads = NoOp>
__device__ void rms_norm_multi_to_smem(int njobs, int n, double inv_n, float eps, float* red, JobFn job,
                                       Layout layout, AfterLoads after_loads = AfterLoads{}) {
  constexpr int NW = NT / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    // One or two vectors of up to 2 * NT 16-byte pieces (the single-sequence kernels): each
    // thread keeps its x and w pieces in registers from the first pass to the second. By the
    // second pass the shared memory is mostly stage buffers, L1 no longer holds x, and
    // re-reading it behind the weight stream took several us.
    constexpr int KC = 2;
    const NormJob J0 = job(0);
    const NormJob J1 = njobs > 1 ? job(1) : NormJob{nullptr, nullptr, nullptr, false};
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    const bool fits = njobs <= 2 && (n & 7) == 0 && n / 8 <= KC * NT && (!J0.valid || (al(J0.x) && al(J0.w))) &&
                      (!J1.valid || (al(J1.x) && al(J1.w)));
    if (fits) {
      const int nv = n / 8;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      uint4 xq[2][KC], wq[2][KC];
#pragma unroll
      for (int i = 0; i < KC; ++i) {
        const int v = tid + i * NT;
        xq[0][i] = (J0.valid && v < nv) ? reinterpret_cast<const uint4*>(J0.x)[v] : z;
        xq[1][i] = (J1.valid && v < nv) ? reinterpret_cast<const uint4*>(J1.x)[v] : z;
        wq[0][i] = (J0.valid && v < nv) ? reinterpret_cast<const uint4*>(J0.w)[v] : z;
        wq[1][i] = (J1.valid && v < nv) ? reinterpret_cast<const uint4*>(J1.w)[v] : z;
      }
      DF acc[2] = {DF{0.0f, 0.0f}, DF{0.0f, 0.0f}};
#pragma unroll
      for (int jj = 0; jj < 2; ++jj)
#pragma unroll
        for (int i = 0; i < KC; ++i) {
          const uint32_t u[4] = {xq[jj][i].x, xq[jj][i].y, xq[jj][i].z, xq[jj][i].w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float a = bf16_lo(u[t]), b = bf16_hi(u[t]);
            df_add(acc[jj], __fmul_rn(a, a));
            df_add(acc[jj], __fmul_rn(b, b));
          }
        }
      after_loads();
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) {
        acc[0] = df_add(acc[0], shfl_xor_df(acc[0], m));
        acc[1] = df_add(acc[1], shfl_xor_df(acc[1], m));
      }
      if (lane == 0)
        for (int jj = 0; jj < njobs; ++jj) {
          red[(jj * NW + warp) * 2] = acc[jj].hi;
          red[(jj * NW + warp) * 2 + 1] = acc[jj].lo;
        }
      __syncthreads();
      float* rr = red + njobs * NW * 2;
      if (tid < njobs) {
        DF tot{red[tid * NW * 2], red[tid * NW * 2 + 1]};
        for (int i = 1; i < NW; ++i) tot = df_add(tot, DF{red[(tid * NW + i) * 2], red[(tid * NW + i) * 2 + 1]});
        // 1 / rms in fp64 (rsqrt: within an ulp or two of the correctly rounded value)
        const double ms = (static_cast<double>(tot.hi) + static_cast<double>(tot.lo)) * inv_n;
        const double r = rsqrt(ms + static_cast<double>(eps));
        const float rh = static_cast<float>(r);
        rr[2 * tid] = rh;
        rr[2 * tid + 1] = static_cast<float>(r - static_cast<double>(rh));
      }
      __syncthreads();
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        if (jj < njobs) {
          const NormJob J = jj == 0 ? J0 : J1;
          const float rh = rr[2 * jj], rl = rr[2 * jj + 1];
#pragma unroll
          for (int i = 0; i < KC; ++i) {
            const int v = tid + i * NT;
            if (v < nv) {
              uint4 o = z;
              if (J.valid) {
                const uint32_t xu[4] = {xq[jj][i].x, xq[jj][i].y, xq[jj][i].z, xq[jj][i].w};
                const uint4 w4 = wq[jj][i];
                const float wf[8] = {bf16_lo(w4.x), bf16_hi(w4.x), bf16_lo(w4.y), bf16_hi(w4.y),
                                     bf16_lo(w4.z), bf16_hi(w4.z), bf16_lo(w4.w), bf16_hi(w4.w)};
                o = bf16x8_scaled_rne(xu, wf, rh, rl);
              }
              // 8 consecutive elements starting at a multiple of 8 stay consecutive in every layout
              *reinterpret_cast<uint4*>(J.out + layout(8 * v)) = o;
            }
          }
        }
      }
      return;
    }
  }
  // Sums of squares, two vectors at a time with their loads in flight together (one memory
  // round trip per pair, not per vector), software-pipelined by one step; the weight vectors
  // are prefetched into L2 alongside (the second pass reads them). after_loads() runs once the
  // first pair has been read: the caller can start its own heavy traffic then, without
  // putting it in front of these reads.
  bool called = false;
  for (int j0 = 0; j0 < njobs; j0 += 2) {
    const NormJob J0 = job(j0);
    const NormJob J1 = (j0 + 1 < njobs) ? job(j0 + 1) : NormJob{nullptr, nullptr, nullptr, false};
    auto vec_ok = [n](const NormJob& J) {
      return !J.valid || (((n & 7) == 0) && ((reinterpret_cast<uintptr_t>(J.x) & 15u) == 0));
    };
    DF acc0{0.0f, 0.0f}, acc1{0.0f, 0.0f};
    if (vec_ok(J0) && vec_ok(J1)) {
      const uint4* x0 = reinterpret_cast<const uint4*>(J0.x);
      const uint4* x1 = reinterpret_cast<const uint4*>(J1.x);
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      const int nv = n / 8;
      int v = tid;
      uint4 q0 = z, q1 = z;
      if (v < nv) {
        if (J0.valid) q0 = x0[v];
        if (J1.valid) q1 = x1[v];
      }
      for (int vw = tid * 8; vw < nv; vw += NT * 8) {  // one 128-byte line of each weight vector
        if (J0.valid) asm volatile("prefetch.global.L2 [%0];" ::"l"(J0.w + 8 * vw));
        if (J1.valid) asm volatile("prefetch.global.L2 [%0];" ::"l"(J1.w + 8 * vw));
      }
      auto sq = [](DF& acc, const uint4& q) {
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float a = bf16_lo(u[t]), b = bf16_hi(u[t]);
          df_add(acc, __fmul_rn(a, a));
          df_add(acc, __fmul_rn(b, b));
        }
      };
      while (v < nv) {
        const int vn = v + NT;
        uint4 n0 = z, n1 = z;
        if (vn < nv) {
          if (J0.valid) n0 = x0[vn];
          if (J1.valid) n1 = x1[vn];
        }
        sq(acc0, q0);
        sq(acc1, q1);
        q0 = n0;
        q1 = n1;
        v = vn;
      }
    } else {
      for (int k = tid; k < n; k += NT) {
        if (J0.valid) {
          const float a = bf16_bits_to_f32(J0.x[k]);
          df_add(acc0, __fmul_rn(a, a));
        }
        if (J1.valid) {
          const float a = bf16_bits_to_f32(J1.x[k]);
          df_add(acc1, __fmul_rn(a, a));
        }
      }
    }
    if (!called) {
      after_loads();
      called = true;
    }
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
      acc0 = df_add(acc0, shfl_xor_df(acc0, m));
      acc1 = df_add(acc1, shfl_xor_df(acc1, m));
    }
    if (lane == 0) {
      red[(j0 * NW + warp) * 2] = acc0.hi;
      red[(j0 * NW + warp) * 2 + 1] = acc0.lo;
      if (j0 + 1 < njobs) {
        red[((j0 + 1) * NW + warp) * 2] = acc1.hi;
        red[((j0 + 1) * NW + warp) * 2 + 1] = acc1.lo;
      }
    }
  }
  if (!called) after_loads();
  __syncthreads();
  float* rr = red + njobs * NW * 2;
  for (int j = tid; j < njobs; j += NT) {
    DF tot{red[j * NW * 2], red[j * NW * 2 + 1]};
    for (int i = 1; i < NW; ++i) tot = df_add(tot, DF{red[(j * NW + i) * 2], red[(j * NW + i) * 2 + 1]});
    // 1 / rms in fp64 (rsqrt: within an ulp or two of the correctly rounded value)
    const double ms = (static_cast<double>(tot.hi) + static_cast<double>(tot.lo)) * inv_n;
    const double r = rsqrt(ms + static_cast<double>(eps));
    const float rh = static_cast<float>(r);
    rr[2 * j] = rh;
    rr[2 * j + 1] = static_cast<float>(r - static_cast<double>(rh));
  }
  __syncthreads();
  for (int j = 0; j < njobs; ++j) {
    const NormJob J = job(j);
    const float rh = rr[2 * j], rl = rr[2 * j + 1];
    const bool vec = ((n & 7) == 0) && ((reinterpret_cast<uintptr_t>(J.x) & 15u) == 0) &&
                     ((reinterpret_cast<uintptr_t>(J.w) & 15u) == 0);
    if (vec) {
      for (int v = tid; v < n / 8; v += NT) {
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (J.valid) {
          const uint4 xq = reinterpret_cast<const uint4*>(J.x)[v];
          const uint4 wq = reinterpret_cast<const uint4*>(J.w)[v];
          const uint32_t xu[4] = {xq.x, xq.y, xq.z, xq.w};
          const float wf[8] = {bf16_lo(wq.x), bf16_hi(wq.x), bf16_lo(wq.y), bf16_hi(wq.y),
                               bf16_lo(wq.z), bf16_hi(wq.z), bf16_lo(wq.w), bf16_hi(wq.w)};
          o = bf16x8_scaled_rne(xu, wf, rh, rl);
        }
        // 8 consecutive elements starting at a multiple of 8 stay consecutive in every layout
        *reinterpret_cast<uint4*>(J.out + layout(8 * v)) = o;
      }
    } else {
      for (int k = tid; k < n; k += NT) {
        uint16_t o = 0;
        if (J.valid) {
          o = static_cast<uint16_t>(
              bf16_scaled_rne(__fmul_rn(bf16_bits_to_f32(J.x[k]), bf16_bits_to_f32(J.w[k])), rh, rl));
        }
        J.out[layout(k)] = o;
      }
    }
  }
}

// Sums of squares of nvec BF16 rows of n elements (n % 8 == 0, rows 16-byte aligned) as
// double-floats (exact squares, TwoSum), for the batched kernels' norm prologues. Threads
// 0..NT-1 call it (NT a multiple of 32; they synchronise on named barrier `bar`). A row is shared
// by tpv threads, tpv the largest power of two with tpv * nvec <= NT; each thread loads kBatch
// 16-byte vectors at a time (independent loads in flight), the tpv partials are combined by a
// fixed shuffle butterfly (within a warp) and, when tpv > 32, the warp totals in warp order --
// the result does not depend on timing. row(j) gives row j (nullptr: a zero row). With kMax it
// also returns max_k |x_k * w_k| (exact products) for the weight vector w. part / mpart: NT / 32
// scratch entries; out / mout: nvec results.
template <int NT, int kBatch, bool kMax, class RowFn>
__device__ void sumsq_rows(int nvec, int n, RowFn row, const uint16_t* w, DF* part, float* mpart, DF* out,
                           float* mout, int bar) {
  const int tid = threadIdx.x, lane = tid & 31;
  int tpv = 1;
  while (tpv * 2 * nvec <= NT) tpv *= 2;
  const int j = tid / tpv, r = tid - j * tpv;
  const int nv = n >> 3;
  DF acc{0.0f, 0.0f};
  float mx = 0.0f;
  if (j < nvec) {
    const uint4* src = reinterpret_cast<const uint4*>(row(j));
    const uint4* wv = reinterpret_cast<const uint4*>(w);
    if (src != nullptr) {
      for (int v0 = r; v0 < nv; v0 += kBatch * tpv) {
        uint4 q[kBatch], wq[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int v = v0 + i * tpv;
          q[i] = v < nv ? src[v] : make_uint4(0u, 0u, 0u, 0u);
          if constexpr (kMax) wq[i] = v < nv ? wv[v] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const uint32_t u[4] = {q[i].x, q[i].y, q[i].z, q[i].w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float lo = bf16_lo(u[t]), hi = bf16_hi(u[t]);
            df_add(acc, __fmul_rn(lo, lo));
            df_add(acc, __fmul_rn(hi, hi));
          }
          if constexpr (kMax) {
            const uint32_t wu[4] = {wq[i].x, wq[i].y, wq[i].z, wq[i].w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              mx = fmaxf(mx, fabsf(__fmul_rn(bf16_lo(u[t]), bf16_lo(wu[t]))));
              mx = fmaxf(mx, fabsf(__fmul_rn(bf16_hi(u[t]), bf16_hi(wu[t]))));
            }
          }
        }
      }
    }
  }
  // butterfly over the row's threads inside the warp (all lanes take part; groups are aligned)
  const int span = tpv < 32 ? tpv : 32;
  for (int m = span >> 1; m > 0; m >>= 1) {
    acc = df_add(acc, shfl_xor_df(acc, m));
    if constexpr (kMax) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
  }
  if (tpv <= 32) {
    if (r == 0 && j < nvec) {
      out[j] = acc;
      if constexpr (kMax) mout[j] = mx;
    }
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(NT) : "memory");
  } else {
    if (lane == 0) {
      part[tid >> 5] = acc;
      if constexpr (kMax) mpart[tid >> 5] = mx;
    }
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(NT) : "memory");
    const int wpv = tpv >> 5;  // warps per row
    if (tid < nvec) {
      DF tot = part[tid * wpv];
      float m = kMax ? mpart[tid * wpv] : 0.0f;
      for (int i = 1; i < wpv; ++i) {
        tot = df_add(tot, part[tid * wpv + i]);
        if constexpr (kMax) m = fmaxf(m, mpart[tid * wpv + i]);
      }
      out[tid] = tot;
      if constexpr (kMax) mout[tid] = m;
    }
  }
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(NT) : "memory");
}

// Shared-memory index of element k of a vector when weight vectors hold 16 elements (FP8) and
// a lane reads the matching 32 bytes of BF16 activations as two 16-byte slots: slots of 32
// consecutive weight vectors are interleaved so both reads of a warp are conflict-free.
struct LayoutIdentity {
  __device__ __forceinline__ int operator()(int k) const { return k; }
};
struct LayoutFp8 {
  __device__ __forceinline__ int operator()(int k) const {
    const int J = k >> 4, e = k & 15;
    const int slot = (J >> 5) * 64 + ((e >> 3) << 5) + (J & 31);
    return slot * 8 + (e & 7);
  }
};

}  // namespace mtp
