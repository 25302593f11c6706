// Exchange key of a vocabulary-shard pick (host and device).
//
// The source's sharded head ("glm5next_mtp_head.rs", `forward_one`, sharded branch) has every
// rank sweep its own row range of lm_head, then combines the ranks' (max logit, index) pairs
// with a SUM all-reduce over eight BF16 lanes, in which `>=` lets the lower rank win a tie.
// Here a pick is one signed 64-bit integer whose order is the argmax order -- the larger
// value first, then the lower global index -- so the pick over any number of shards is the
// plain maximum of their keys: one MAX reduction (or one kernel over R keys), exact, with the
// FP32 value intact.
//
//   bits 63..32  the value's IEEE bits mapped to an unsigned order: a negative value has all its
//                bits inverted, a non-negative one gets the sign bit set; -0 is taken as +0,
//                since the argmax treats the two as equal
//   bits 31..0   the bitwise complement of the global index, so a lower index gives a larger key
//   then bit 63 is flipped, which turns the unsigned order into the signed order of int64.
//
// The empty pick (no rows, or every logit NaN) is INT64_MIN; it decodes to index -1 and is
// below every real key (a real key's upper half is at least that of -inf, 0x007FFFFF, and its
// lower half at least 0x80000000). NaN never gets a key of its own.
#pragma once

#include <stdint.h>

#ifdef __CUDACC__
#define MTP_PICK_FN __host__ __device__ __forceinline__
#else
#define MTP_PICK_FN static inline
#endif

namespace mtp {

constexpr int64_t kPickEmpty = -0x7FFFFFFFFFFFFFFFLL - 1;

MTP_PICK_FN uint32_t pick_float_bits(float v) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(v);
#else
  union {
    float f;
    uint32_t u;
  } c;
  c.f = v;
  return c.u;
#endif
}

MTP_PICK_FN float pick_bits_float(uint32_t u) {
#ifdef __CUDA_ARCH__
  return __uint_as_float(u);
#else
  union {
    float f;
    uint32_t u;
  } c;
  c.u = u;
  return c.f;
#endif
}

// Key of (value, global index); kPickEmpty when index < 0 or value is NaN.
MTP_PICK_FN int64_t pick_key(float value, int32_t index) {
  if (index < 0 || value != value) return kPickEmpty;
  uint32_t u = pick_float_bits(value);
  if ((u & 0x7FFFFFFFu) == 0u) u = 0u;
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  const uint64_t k = (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(~static_cast<uint32_t>(index));
  return static_cast<int64_t>(k ^ 0x8000000000000000ull);
}

// Global index of a key (-1 for the empty key).
MTP_PICK_FN int32_t pick_index(int64_t key) {
  return static_cast<int32_t>(~static_cast<uint32_t>(static_cast<uint64_t>(key)));
}

// Value of a key (NaN for the empty key; +0 for a pick made from -0).
MTP_PICK_FN float pick_value(int64_t key) {
  const uint32_t ord = static_cast<uint32_t>((static_cast<uint64_t>(key) ^ 0x8000000000000000ull) >> 32);
  return pick_bits_float((ord & 0x80000000u) ? (ord & 0x7FFFFFFFu) : ~ord);
}

}  // namespace mtp
