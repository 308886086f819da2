// Row-level helpers shared by the sampler and the verifier: order-key widths,
// 16-byte vector operations, the row maximum, and the exact top-p target.
#pragma once

#include "common.cuh"

namespace smp {

// Key width per element type: bf16 keys are the upper 16 bits of the binary32 key.
template <typename T>
struct KeyTraits;
template <>
struct KeyTraits<float> {
  static constexpr int kBits = 32;
  static constexpr int kLevels = 4;
};
template <>
struct KeyTraits<uint16_t> {
  static constexpr int kBits = 16;
  static constexpr int kLevels = 2;
};

// Operations on one 16-byte vector of elements: packed maximum, element access.
template <typename T>
struct VecOps;

template <>
struct VecOps<uint16_t> {
  static constexpr int kPer = 8;
  static __device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  static __device__ __forceinline__ uint32_t neg_inf() { return 0xFF80FF80u; }
  // max of the 8 values of x, packed in two halves
  static __device__ __forceinline__ uint32_t vmax(const uint4& x) {
    return max2(max2(x.x, x.y), max2(x.z, x.w));
  }
  static __device__ __forceinline__ float finish(uint32_t m) {
    return fmaxf(__uint_as_float(m & 0xFFFF0000u), __uint_as_float(m << 16));
  }
  // element q (0..7, a compile-time constant once unrolled) of x
  static __device__ __forceinline__ float elem(const uint4& x, int q) {
    const uint32_t w = q < 2 ? x.x : q < 4 ? x.y : q < 6 ? x.z : x.w;
    return __uint_as_float((q & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
  // The threshold for ge_mask: the smallest bf16 value >= theta, in both
  // halves (a bf16 element is >= theta exactly when it is >= that value).
  static __device__ __forceinline__ uint32_t threshold(float theta) {
    const uint32_t b = __float_as_uint(theta);
    if ((b & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC07FC0u;   // NaN: no element qualifies
    uint32_t h = b >> 16;
    if ((b & 0xFFFFu) && !(b & 0x80000000u)) ++h;   // positive and inexact: round up
    return h | (h << 16);                            // (negative: truncation rounds up)
  }
  // Bit q set when element q of x >= the threshold (NaN elements never).
  static __device__ __forceinline__ uint32_t ge_mask(const uint4& x, uint32_t t) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t r;
      asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(w[i]), "r"(t));
      m |= ((r & 1u) << (2 * i)) | (((r >> 16) & 1u) << (2 * i + 1));
    }
    return m;
  }
};

template <>
struct VecOps<float> {
  static constexpr int kPer = 4;
  static __device__ __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    return __float_as_uint(fmaxf(__uint_as_float(a), __uint_as_float(b)));
  }
  static __device__ __forceinline__ uint32_t neg_inf() { return 0xFF800000u; }
  static __device__ __forceinline__ uint32_t vmax(const uint4& x) {
    return __float_as_uint(fmaxf(fmaxf(__uint_as_float(x.x), __uint_as_float(x.y)),
                                 fmaxf(__uint_as_float(x.z), __uint_as_float(x.w))));
  }
  static __device__ __forceinline__ float finish(uint32_t m) { return __uint_as_float(m); }
  static __device__ __forceinline__ float elem(const uint4& x, int q) {
    return __uint_as_float(q == 0 ? x.x : q == 1 ? x.y : q == 2 ? x.z : x.w);
  }
  static __device__ __forceinline__ uint32_t threshold(float theta) { return __float_as_uint(theta); }
  static __device__ __forceinline__ uint32_t ge_mask(const uint4& x, uint32_t t) {
    const float th = __uint_as_float(t);
    return (__uint_as_float(x.x) >= th ? 1u : 0u) | (__uint_as_float(x.y) >= th ? 2u : 0u) |
           (__uint_as_float(x.z) >= th ? 4u : 0u) | (__uint_as_float(x.w) >= th ? 8u : 0u);
  }
};

__device__ __forceinline__ float block_max_f(float v, float* scratch) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  cta_sync();
  if (lane == 0) scratch[warp] = v;
  cta_sync();
  float r = scratch[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) r = fmaxf(r, scratch[w]);
  return r;
}

template <typename T>
__device__ __forceinline__ float key_value(uint32_t key) {
  if (KeyTraits<T>::kBits == 32) return value_of_key(key);
  const uint32_t fill = (key & 0x8000u) ? 0u : 0xFFFFu;
  return value_of_key((key << 16) | fill);
}

template <typename T>
__device__ __forceinline__ bool key_finite(uint32_t key) {
  return KeyTraits<T>::kBits == 32 ? key_is_finite(key) : key_is_finite((key << 16) | ((key & 0x8000u) ? 0u : 0xFFFFu));
}

// Target of a mass select: the prefix reaches top_p * Z  <=>  (H << sh) >= rhs.
struct MassTarget {
  u128 rhs;
  int sh;
  bool trivial;   // top_p so small that one token always suffices
};

__device__ __forceinline__ MassTarget make_mass_target(float top_p, uint64_t z_total) {
  MassTarget t;
  t.trivial = false;
  t.sh = 0;
  t.rhs = 0;
  if (!(top_p > 0.0f)) {
    t.trivial = true;
    return t;
  }
  const uint32_t b = __float_as_uint(top_p);
  int ex = int((b >> 23) & 0xFF);
  uint32_t mant = b & 0x7FFFFFu;
  if (ex == 0) {
    t.trivial = true;   // subnormal top_p: any single token reaches it
    return t;
  }
  mant |= 0x800000u;
  const int e2 = ex - 127 - 23;        // top_p = mant * 2^e2, e2 <= -24 for top_p < 1
  if (-e2 > 100) {
    t.trivial = true;
    return t;
  }
  t.sh = -e2;                          // H * 2^sh >= mant * Z
  if (t.sh > 63) {
    // Z <= 2^63 and H >= 2^44 for the first token: top_p < 2^-40 always holds at one token.
    t.trivial = true;
    return t;
  }
  t.rhs = u128(mant) * z_total;
  return t;
}

__device__ __forceinline__ bool mass_reaches(uint64_t h, const MassTarget& t) {
  return (u128(h) << t.sh) >= t.rhs;
}

}  // namespace smp
