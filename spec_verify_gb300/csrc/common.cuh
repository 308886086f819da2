// Device building blocks shared by the sampler and verifier kernels:
// logit keys, Philox4x64-10, the fixed-point probability mass, block and
// cluster reductions, DSMEM mailboxes and bounded waits.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "exp_table.h"

namespace smp {

constexpr int kThreads = 256;                 // threads per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kFixedBits = 44;                // E = round(e * 2^44)
constexpr uint64_t kFixedOne = 1ull << kFixedBits;

// Row status flags (mirror SMP_ROW_* of smp.h).
constexpr int kRowBadParams = 1;
constexpr int kRowNonFinite = 2;
constexpr int kRowTimeout = 4;
constexpr int kRowBadDraft = 8;

typedef unsigned __int128 u128;

// ------------------------------------------------------------------ keys
//
// The order of logits is the order of 32-bit keys: for a float's bits b,
// key = b | 0x80000000 for non-negative values and ~b for negative ones.
// NaN takes the key of -inf and -0 the key of +0, so ties and NaNs behave as
// the oracle's float comparisons do.  bf16 logits are widened to binary32.

constexpr uint32_t kKeyNegInf = 0x007FFFFFu;
constexpr uint32_t kKeyPosInf = 0xFF800000u;

__device__ __forceinline__ uint32_t key_of_bits(uint32_t b) {
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) b = 0xFF800000u;   // NaN -> -inf
  if (b == 0x80000000u) b = 0u;                           // -0 -> +0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float value_of_key(uint32_t key) {
  uint32_t b = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
  return __uint_as_float(b);
}

__device__ __forceinline__ bool key_is_finite(uint32_t key) {
  return key > kKeyNegInf && key < kKeyPosInf;
}

// Elements of a row, as stored in shared memory.
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static __device__ __forceinline__ uint32_t bits(float v) { return __float_as_uint(v); }
  static __device__ __forceinline__ float widen(float v) { return v; }
};

template <>
struct Elem<uint16_t> {   // bf16 bit pattern
  static __device__ __forceinline__ uint32_t bits(uint16_t v) { return uint32_t(v) << 16; }
  static __device__ __forceinline__ float widen(uint16_t v) { return __uint_as_float(uint32_t(v) << 16); }
};

// ------------------------------------------------------------------ Philox4x64-10
//
// Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11): 10 rounds of (c0, c1, c2, c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
// hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)) with a Weyl key schedule between rounds.

__device__ __forceinline__ uint64_t philox_word0(uint64_t seed, uint64_t offset,
                                                 uint64_t row, uint64_t draw) {
  const uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
  const uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
  uint64_t c0 = offset, c1 = row, c2 = draw, c3 = 0;
  uint64_t k0 = seed, k1 = 0;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint64_t hi0 = __umul64hi(kM0, c0), lo0 = kM0 * c0;
    const uint64_t hi1 = __umul64hi(kM1, c2), lo1 = kM1 * c2;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
  }
  return c0;
}

// The 53-bit integer U with u = U * 2^-53.
__device__ __forceinline__ uint64_t uniform53(uint64_t seed, uint64_t offset, uint64_t row,
                                              uint64_t draw) {
  return philox_word0(seed, offset, row, draw) >> 11;
}

// ------------------------------------------------------------------ double-float exponential
//
// e = exp(x) for x = (z - m) * (1/T), evaluated in pairs of binary32 numbers
// (head + tail) after the table-driven method of P. T. P. Tang, "Table-driven
// implementation of the exponential function in IEEE floating-point
// arithmetic", ACM TOMS 15(2), 1989: y = x log2(e) = n + j/64 + f, |f| <= 1/128,
// e = 2^n * 2^(j/64) * exp(f ln 2), with 2^(j/64) from a 64-entry table and
// exp(g) - 1 from its Taylor series to degree 5 (|g| < 0.0055, truncation below
// 2^-54).  Exact sums and products use the error-free transformations TwoSum
// (Knuth) and TwoProduct through a fused multiply-add.  Relative error stays
// below about 2^-46, far inside the 2^-44 grid of the fixed-point masses.

struct RowScale {
  float m;        // row maximum logit
  float c_hi;     // c = log2(e) / T as a head ...
  float c_lo;     // ... and tail
};

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// c = log2(e) / T as head + tail, in binary32 arithmetic: q = L_hi / T, then
// the exact residual L_hi - q T (one fused multiply-add) plus L_lo, divided by T.
__device__ __forceinline__ RowScale make_row_scale(float m, float temperature) {
  constexpr float kLog2eHi = 0x1.715476p+0f;     // binary32 nearest log2(e)
  constexpr float kLog2eLo = 0x1.4ae0cp-26f;     // log2(e) - kLog2eHi
  RowScale rs;
  rs.m = m;
  const float q = __fdiv_rn(kLog2eHi, temperature);
  const float r = __fadd_rn(__fmaf_rn(-q, temperature, kLog2eHi), kLog2eLo);
  rs.c_hi = q;
  rs.c_lo = __fdiv_rn(r, temperature);
  return rs;
}

// make_row_scale(m, 1) without the divisions: c = log2(e) as head + tail.
__device__ __forceinline__ RowScale make_row_scale_unit(float m) {
  RowScale rs;
  rs.m = m;
  rs.c_hi = 0x1.715476p+0f;
  rs.c_lo = 0x1.4ae0cp-26f;
  return rs;
}

// Result of the exponential before scaling: e = (hi + lo) * 2^n, hi in [~0.98, ~2.03).
struct ExpParts {
  float hi;
  float lo;
  int n;
  int kind;   // 0: regular; 1: exactly 1 (z == m); 2: zero (below the fixed-point grid)
};

// exp((z - m) / T) for z <= m.  Returns kind 2 when log2 of the value is
// below `ymin`.
__device__ __forceinline__ ExpParts exp_parts(float z, const RowScale& rs, const FloatPair* table,
                                              float ymin) {
  ExpParts out;
  out.hi = 1.0f;
  out.lo = 0.0f;
  out.n = 0;
  out.kind = 0;
  float d_hi, d_lo;
  two_sum(z, -rs.m, d_hi, d_lo);            // d = z - m exactly
  if (d_hi == 0.0f) {
    out.kind = 1;
    return out;
  }
  const float y_hi = __fmul_rn(d_hi, rs.c_hi);
  if (!(y_hi > ymin)) {                     // also catches -inf and NaN
    out.kind = 2;
    return out;
  }
  const float y_lo = __fadd_rn(__fmaf_rn(d_hi, rs.c_hi, -y_hi),
                               __fmaf_rn(d_hi, rs.c_lo, __fmul_rn(d_lo, rs.c_hi)));
  const float kf = rintf(__fmul_rn(y_hi, 64.0f));
  const int k = int(kf);
  const float r = __fmaf_rn(kf, -0.015625f, y_hi);   // y_hi - k/64, exact
  float f_hi, f_lo;
  two_sum(r, y_lo, f_hi, f_lo);                     // f = y - k/64
  // g = f * ln 2
  const float g_hi = __fmul_rn(f_hi, kLn2Hi);
  const float g_lo = __fadd_rn(__fmaf_rn(f_hi, kLn2Hi, -g_hi),
                               __fmaf_rn(f_hi, kLn2Lo, __fmul_rn(f_lo, kLn2Hi)));
  // exp(g) - 1 = g + g^2/2 + g^3/6 + g^4/24 + g^5/120
  const float s2_hi = __fmul_rn(g_hi, g_hi);
  const float s2_lo = __fmaf_rn(g_hi, g_hi, -s2_hi);
  const float poly = __fmaf_rn(g_hi, __fmaf_rn(g_hi, 1.0f / 120.0f, 1.0f / 24.0f), 1.0f / 6.0f);
  const float c3 = __fmul_rn(__fmul_rn(s2_hi, g_hi), poly);
  const float small = __fadd_rn(__fadd_rn(g_lo, __fmaf_rn(g_hi, g_lo, __fmul_rn(0.5f, s2_lo))),
                                __fmaf_rn(__fmul_rn(0.5f, s2_hi), g_lo, c3));
  float em_hi, em_lo;
  two_sum(g_hi, __fmul_rn(0.5f, s2_hi), em_hi, em_lo);
  em_lo = __fadd_rn(em_lo, small);
  // multiply by 2^(j/64) = t_hi + t_lo
  const FloatPair t = table[k & 63];
  const float p_hi = __fmul_rn(t.hi, em_hi);
  const float p_lo = __fmaf_rn(t.hi, em_hi, -p_hi);
  float r_hi, r_lo;
  two_sum(t.hi, p_hi, r_hi, r_lo);
  const float tail = __fadd_rn(__fadd_rn(p_lo, __fmul_rn(t.hi, em_lo)),
                               __fmaf_rn(t.lo, em_hi, t.lo));
  r_lo = __fadd_rn(r_lo, tail);
  out.hi = r_hi;
  out.lo = r_lo;
  out.n = k >> 6;   // floor(k / 64)
  return out;
}

// 2^s as a float for s in [-126, 127].
__device__ __forceinline__ float pow2f(int s) { return __int_as_float((s + 127) << 23); }

// The fixed-point mass E = round(e * 2^F) of an exponential in parts.
__device__ __forceinline__ uint64_t fixed_from_parts(const ExpParts& e) {
  if (e.kind == 1) return kFixedOne;
  if (e.kind == 2) return 0;
  const int s = kFixedBits + e.n;           // E = (hi + lo) * 2^s
  if (s < -2) return 0;
  const float sc = pow2f(s);
  const float hs = __fmul_rn(e.hi, sc);     // exact
  const float ls = __fmul_rn(e.lo, sc);     // exact
  if (s >= 25) {
    // hs is an integer >= 2^24: take it from its bits, then add the rounded tail.
    const uint32_t b = __float_as_uint(hs);
    const uint64_t mant = uint64_t((b & 0x7FFFFFu) | 0x800000u);
    const int sh = int((b >> 23) & 0xFF) - 127 - 23;
    const uint64_t head = mant << sh;
    // |lo| <= ulp(hi): |ls| < 2^22 for s <= F, so a 32-bit conversion suffices
    // (64-bit float-to-integer conversions are slower on this part).
    const int t = __float2int_rn(ls);
    return uint64_t((long long)head + t);
  }
  const float v = rintf(__fadd_rn(hs, ls));      // an integer below 2^25
  return v <= 0.0f ? 0ull : uint64_t(__float2uint_rz(v));
}

// An exponential in parts as a double (head + tail, scaled).
__device__ __forceinline__ double double_from_parts(const ExpParts& e) {
  if (e.kind == 1) return 1.0;
  if (e.kind == 2) return 0.0;
  return ldexp(double(e.hi) + double(e.lo), e.n);
}

// The fixed-point mass E = round(exp((z - m) / T) * 2^F).
__device__ __forceinline__ uint64_t mass_fixed(float z, const RowScale& rs, const FloatPair* table) {
  return fixed_from_parts(exp_parts(z, rs, table, -float(kFixedBits + 3)));
}

// 2^y by the ex2.approx instruction (flushes results below 2^-126 to 0).
__device__ __forceinline__ float ex2_approx(float y) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}

// exp((z - m) / T) in binary32 (0 for -inf, NaN and below 2^-126).
__device__ __forceinline__ float exp_fast(float z, const RowScale& rs) {
  const float d = __fsub_rn(z, rs.m);
  const float y = __fmaf_rn(d, rs.c_hi, __fmul_rn(d, rs.c_lo));
  return y > -126.0f ? ex2_approx(y) : 0.0f;
}

// (hi + lo) * 2^n >= x for an exponential in parts and 0 < x < 1, exactly,
// in binary32: hi * 2^n and lo * 2^n are exact for n >= -100, and within a
// factor of two of x the difference hi * 2^n - x is exact (Sterbenz), so its
// sum with lo * 2^n has the sign of the comparison.
__device__ __forceinline__ bool parts_at_least(const ExpParts& e, float x) {
  if (e.kind == 1) return true;
  if (e.kind == 2) return false;
  if (e.n < -100) return double_from_parts(e) >= double(x);
  const float sc = pow2f(e.n);
  const float vh = __fmul_rn(e.hi, sc), vl = __fmul_rn(e.lo, sc);
  if (vh >= __fmul_rn(2.0f, x)) return true;
  if (__fmul_rn(2.0f, vh) < x) return false;
  return __fsub_rn(vh, x) >= -vl;
}

// exp((z - m) / T) as a double (head + tail, scaled); 0 below 2^-1000.
__device__ __forceinline__ double mass_double(float z, const RowScale& rs, const FloatPair* table) {
  return double_from_parts(exp_parts(z, rs, table, -1000.0f));
}

// ------------------------------------------------------------------ warp / block helpers

// Programmatic dependent launch: wait until the previous kernel on the stream
// has finished and its writes are visible (a no-op for a normal launch), and
// let the next kernel on the stream be scheduled early (it waits in turn).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// Barrier over the kThreads threads that work on rows (named barrier 1).  A
// kernel may run an extra producer warp that takes no part in it.
__device__ __forceinline__ void cta_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

// A global word written earlier in this kernel (by this CTA, before a barrier).
__device__ __forceinline__ int32_t load_volatile(const int32_t* p) { return *reinterpret_cast<const volatile int32_t*>(p); }

// cta_sync() that also returns how many of the kThreads threads passed `pred`.
__device__ __forceinline__ int cta_sync_count(bool pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.popc.u32 %0, 1, %2, q;\n\t}"
      : "=r"(r)
      : "r"(int(pred)), "n"(kThreads)
      : "memory");
  return r;
}

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int mask) {
  const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, uint32_t(v), mask);
  const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, uint32_t(v >> 32), mask);
  return (uint64_t(hi) << 32) | lo;
}

__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(0xFFFFFFFFu, uint32_t(v), src);
  const uint32_t hi = __shfl_sync(0xFFFFFFFFu, uint32_t(v >> 32), src);
  return (uint64_t(hi) << 32) | lo;
}

__device__ __forceinline__ uint64_t shfl_up_u64(uint64_t v, int delta) {
  const uint32_t lo = __shfl_up_sync(0xFFFFFFFFu, uint32_t(v), delta);
  const uint32_t hi = __shfl_up_sync(0xFFFFFFFFu, uint32_t(v >> 32), delta);
  return (uint64_t(hi) << 32) | lo;
}

__device__ __forceinline__ u128 shfl_xor_u128(u128 v, int mask) {
  const uint64_t lo = shfl_xor_u64(uint64_t(v), mask);
  const uint64_t hi = shfl_xor_u64(uint64_t(v >> 64), mask);
  return (u128(hi) << 64) | lo;
}

__device__ __forceinline__ u128 shfl_up_u128(u128 v, int delta) {
  const uint64_t lo = shfl_up_u64(uint64_t(v), delta);
  const uint64_t hi = shfl_up_u64(uint64_t(v >> 64), delta);
  return (u128(hi) << 64) | lo;
}

template <typename U>
__device__ __forceinline__ U warp_sum(U v);

template <>
__device__ __forceinline__ uint32_t warp_sum<uint32_t>(uint32_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

template <>
__device__ __forceinline__ uint64_t warp_sum<uint64_t>(uint64_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += shfl_xor_u64(v, o);
  return v;
}

template <>
__device__ __forceinline__ u128 warp_sum<u128>(u128 v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += shfl_xor_u128(v, o);
  return v;
}

// Inclusive prefix sum over the lanes of a warp.
template <typename U>
__device__ __forceinline__ U warp_inclusive_scan(U v);

template <>
__device__ __forceinline__ uint32_t warp_inclusive_scan<uint32_t>(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

template <>
__device__ __forceinline__ uint64_t warp_inclusive_scan<uint64_t>(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint64_t o = shfl_up_u64(v, d);
    if (lane >= d) v += o;
  }
  return v;
}

template <>
__device__ __forceinline__ u128 warp_inclusive_scan<u128>(u128 v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const u128 o = shfl_up_u128(v, d);
    if (lane >= d) v += o;
  }
  return v;
}

// Largest key, lowest id among equal keys, packed as (key << 32) | ~id.
// Warp-aggregated shared-memory updates.  Every lane of the warp must call
// these together; many lanes hitting one address would otherwise serialise.

__device__ __forceinline__ uint64_t pack_key_id(uint32_t key, uint32_t id) {
  return (uint64_t(key) << 32) | uint64_t(~id);
}

__device__ __forceinline__ uint64_t block_max_u64(uint64_t v, uint64_t* scratch) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const uint64_t w = shfl_xor_u64(v, o);
    v = w > v ? w : v;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  cta_sync();
  if (lane == 0) scratch[warp] = v;
  cta_sync();
  uint64_t best = scratch[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) best = scratch[w] > best ? scratch[w] : best;
  return best;
}

// ------------------------------------------------------------------ cluster plumbing
//
// A row is processed by the CTAs of one thread-block cluster.  Each CTA
// publishes partial results in a mailbox in its own shared memory; after a
// cluster barrier every CTA reads all mailboxes through distributed shared
// memory.  Mailboxes alternate between two buffers, so one barrier per
// exchange is enough.  The barrier is an mbarrier per CTA that every CTA of
// the cluster arrives on remotely; its wait is bounded in time and a timeout
// marks the row (SMP_ROW_TIMEOUT) instead of spinning forever.

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return uint32_t(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ uint64_t ld_cluster_u64(uint32_t addr) {
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_cluster_u64(uint32_t addr, uint64_t v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void hw_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

}  // namespace smp
