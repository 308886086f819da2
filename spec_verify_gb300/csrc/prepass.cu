// Logit pre-pass in place: the repetition penalty ("Choosing the next word",
// section "The repetition penalty": z_i <- z_i / r if z_i > 0, else z_i * r,
// for each distinct token i among the row's recent tokens) and the
// constraint mask ("Decoding & Speculative Sampling", section 39.3: tokens
// outside the allowed set get -inf), written into the caller's logits so that
// smp_sample (or the verifier) then reads them in its own single pass.
//
// Only changed elements are written: -inf at disallowed ids, the penalised
// value at the (at most 64) distinct history ids that are allowed.  The two
// sets are disjoint, so no element is written twice and the result does not
// depend on the order in which CTAs run.
#include <cuda_runtime.h>

#include "launch.h"
#include "row_ops.cuh"
#include "smp.h"

namespace smp {

constexpr int kPrepassWordsPerCta = kWarps * 32;   // 32 mask words (1024 ids) per warp

struct PrepassArgs {
  void* logits;
  int batch;
  int vocab;
  int words;                  // ceil(vocab / 32)
  int chunks;                 // CTAs per row
  const uint32_t* allowed;    // [batch, words] or nullptr
  const int32_t* history;     // [batch, hist_len] or nullptr
  int hist_len;
  const float* penalty;       // [batch] or nullptr
  int32_t* status;
};

template <typename T>
struct Bits;
template <>
struct Bits<float> {
  static constexpr uint32_t kNegInf = 0xFF800000u;
  static constexpr uint32_t kNaN = 0x7FC00000u;
  static __device__ __forceinline__ void store(float* p, uint32_t b) { *reinterpret_cast<uint32_t*>(p) = b; }
  static __device__ __forceinline__ float load(const float* p) { return *p; }
  static __device__ __forceinline__ void store_value(float* p, float z) { *p = z; }
};
template <>
struct Bits<uint16_t> {
  static constexpr uint32_t kNegInf = 0xFF80u;
  static constexpr uint32_t kNaN = 0x7FC0u;
  static __device__ __forceinline__ void store(uint16_t* p, uint32_t b) { *p = uint16_t(b); }
  static __device__ __forceinline__ float load(const uint16_t* p) { return __uint_as_float(uint32_t(*p) << 16); }
  // z is a bf16 value already (rounded by the caller)
  static __device__ __forceinline__ void store_value(uint16_t* p, float z) { *p = uint16_t(__float_as_uint(z) >> 16); }
};

// Nearest bf16 value of a binary32 number (ties to even); NaN and infinities kept.
__device__ __forceinline__ float prepass_round_bf16(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return x;
  b = (b + 0x7FFFu + ((b >> 16) & 1u)) & 0xFFFF0000u;
  return __uint_as_float(b);
}

__device__ __forceinline__ bool allowed_bit(const uint32_t* words, int id) {
  return words == nullptr || ((words[id >> 5] >> (id & 31)) & 1u);
}

// One CTA per (row, chunk of kPrepassWordsPerCta mask words).  Each warp takes
// 32 words: lane l loads word l, then for each word the warp stores -inf at
// its disallowed ids (lane l: id 32 w + l), one coalesced store per word that
// is not all ones.  Chunk 0's warp 0 applies the penalty.  A row whose factor
// r is not finite and > 0 is filled with NaN instead (every chunk its part).
template <typename T>
__global__ void __launch_bounds__(kThreads) logit_prepass_kernel(PrepassArgs a) {
  const int row = int(blockIdx.x) / a.chunks;
  const int chunk = int(blockIdx.x) % a.chunks;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dependency_wait();
  allow_dependent_launch();
  T* z = reinterpret_cast<T*>(a.logits) + size_t(row) * a.vocab;
  const float r = a.penalty ? a.penalty[row] : 1.0f;
  const bool bad = !(isfinite(r) && r > 0.0f);
  const uint32_t* words = a.allowed ? a.allowed + size_t(row) * a.words : nullptr;
  const int w0 = chunk * kPrepassWordsPerCta + warp * 32;

  if (bad) {
    if (chunk == 0 && threadIdx.x == 0 && a.status) atomicOr(a.status, kRowBadParams);
    const int id0 = w0 * 32, id1 = min(a.vocab, (w0 + 32) * 32);
    for (int id = id0 + lane; id < id1; id += 32) Bits<T>::store(z + id, Bits<T>::kNaN);
    return;
  }

  if (words != nullptr && w0 < a.words) {
    const uint32_t mine = w0 + lane < a.words ? words[w0 + lane] : 0xFFFFFFFFu;
    // bits past the vocabulary count as allowed (nothing to write there)
    const int last = a.vocab - (a.words - 1) * 32;   // ids in the last word, 1..32
    const uint32_t tail_ones = last == 32 ? 0u : ~((1u << last) - 1u);
    const uint32_t w = (w0 + lane == a.words - 1) ? (mine | tail_ones) : mine;
    const uint32_t todo = __ballot_sync(0xFFFFFFFFu, w != 0xFFFFFFFFu);
    for (uint32_t m = todo; m; m &= m - 1) {
      const int j = __ffs(m) - 1;
      const uint32_t wj = __shfl_sync(0xFFFFFFFFu, w, j);
      if (!((wj >> lane) & 1u)) Bits<T>::store(z + (w0 + j) * 32 + lane, Bits<T>::kNegInf);
    }
  }

  if (chunk == 0 && warp == 0 && a.history && a.hist_len > 0 && r != 1.0f) {
    // entries lane and lane + 32; an entry is applied at its first occurrence only
    const int H = a.hist_len;
    const int32_t* h = a.history + size_t(row) * H;
    const int32_t e0 = lane < H ? h[lane] : -1;
    const int32_t e1 = lane + 32 < H ? h[lane + 32] : -1;
    bool first0 = e0 >= 0 && e0 < a.vocab, first1 = e1 >= 0 && e1 < a.vocab;
    for (int s = 0; s < 64; ++s) {
      const int32_t o = __shfl_sync(0xFFFFFFFFu, s < 32 ? e0 : e1, s & 31);
      if (s < lane && o == e0) first0 = false;
      if (s < lane + 32 && o == e1) first1 = false;
    }
    auto apply = [&](int32_t id) {
      if (!allowed_bit(words, id)) return;   // the mask writes -inf there
      float v = Bits<T>::load(z + id);
      v = v > 0.0f ? __fdiv_rn(v, r) : __fmul_rn(v, r);
      if (sizeof(T) == 2) v = prepass_round_bf16(v);
      Bits<T>::store_value(z + id, v);
    };
    if (first0) apply(e0);
    if (first1) apply(e1);
  }
}

template <typename T>
static smp_status launch_prepass(const PrepassArgs& args, cudaStream_t stream) {
  PrepassArgs a = args;
  LaunchShape ls;
  ls.pdl = true;
  const int64_t grid = int64_t(a.batch) * a.chunks;
  if (grid > 0x7FFFFFFF) return SMP_ERR_INVALID_ARG;
  const cudaError_t err = launch_cluster(reinterpret_cast<const void*>(&logit_prepass_kernel<T>),
                                         dim3(unsigned(grid)), dim3(kThreads), ls, stream, &a);
  if (err != cudaSuccess) return fail_cuda(err);
  return SMP_OK;
}

}  // namespace smp

extern "C" smp_status smp_logit_prepass(void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                                        const uint32_t* allowed, const int32_t* history, int32_t history_len,
                                        const float* repetition_penalty, int32_t* status, void* stream) {
  using namespace smp;
  if (dtype != SMP_F32 && dtype != SMP_BF16) return SMP_ERR_DTYPE;
  if (!logits || batch <= 0 || vocab <= 0) return SMP_ERR_INVALID_ARG;
  if (vocab > SMP_MAX_VOCAB) return SMP_ERR_UNSUPPORTED;
  if (history_len < 0 || history_len > SMP_MAX_HISTORY || (history_len > 0 && !history))
    return SMP_ERR_INVALID_ARG;
  const int elem = dtype == SMP_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(logits) % elem) return SMP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(allowed) | reinterpret_cast<uintptr_t>(history) |
       reinterpret_cast<uintptr_t>(repetition_penalty) | reinterpret_cast<uintptr_t>(status)) % 4)
    return SMP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (status) {
    const smp_status rc = clear_status(status, st);
    if (rc != SMP_OK) return rc;
  }
  PrepassArgs a{};
  a.logits = logits;
  a.batch = batch;
  a.vocab = vocab;
  a.words = (vocab + 31) / 32;
  a.chunks = (a.words + kPrepassWordsPerCta - 1) / kPrepassWordsPerCta;
  a.allowed = allowed;
  a.history = history_len > 0 ? history : nullptr;
  a.hist_len = history_len;
  a.penalty = repetition_penalty;
  a.status = status;
  if (dtype == SMP_F32) return launch_prepass<float>(a, st);
  return launch_prepass<uint16_t>(a, st);
}
