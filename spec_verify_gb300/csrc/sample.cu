// Batched next-token sampler: temperature, top-k, top-p and min-p, the
// renormalised distribution of eq. 39.2 ("Decoding & Speculative Sampling",
// section 39.2) and an id-order inverse-CDF draw ("Choosing the next word",
// section "Where the randomness comes from, and where it stops").
//
// Rows are independent, so each CTA owns whole rows and no CTA ever waits for
// another.  Two paths, chosen from a row's knobs:
//
//  * candidate path -- greedy rows, min-p rows, and top-k rows with small k
//    (no top-p).  The kept set S is a short prefix of the order (logit
//    descending, id ascending).  The row streams once from HBM through a TMA
//    ring in shared memory; every element at or above a running lower bound
//    of S's boundary becomes a candidate, and S is selected exactly among the
//    candidates at the end of the row.
//
//  * general path -- top-p rows, unfiltered sampling, large k, or a candidate
//    overflow, run by the row's CTA over global memory: for bf16 rows the
//    per-value count table (general_bf16.cuh); else, with top-k up to
//    kTopKMax, a ranked candidate list (select.cuh); else exact radix
//    selection over logit keys; 64-bit fixed-point masses throughout
//    (row_ops.cuh).
//
// All decisions use exact integers (keys, fixed-point masses), so results do
// not depend on how rows are scheduled.
#include <cuda_runtime.h>
#include <stdio.h>

#include "launch.h"
#include "row_ops.cuh"
#include "smp.h"
#include "tma.cuh"

namespace smp {

#include "select.cuh"

constexpr int kBufBytes = 32768;                       // one TMA copy: a batch of the row
constexpr int kBufs = 2;                               // batches in flight per CTA (double buffering)
constexpr int kPrefetchBatches = 8;                    // batches of the first row prefetched into L2
constexpr int kSubBytes = kBufBytes / kWarps;          // the part of a batch one warp processes
constexpr int kVecPerLane = kSubBytes / 16 / 32;       // 16-byte vectors per lane and batch
static_assert(kVecPerLane == 8, "a lane's unit is one 128-byte line, read in XOR-swizzled order");
constexpr int kCandMax = 1024;    // candidate list capacity per row
constexpr int kFinalMax = kThreads;   // candidates at or above the final threshold (one per thread)
constexpr int kSegs = 8;          // segment maxima kept per lane and row (min-p / top-k rows)
constexpr int kFastTopK = 128;    // top-k rows up to this k take the candidate path
// out_ids value that marks a row for the general path at the end of the CTA's
// rows (never a result: results are token ids >= 0, or -1).
constexpr int32_t kHandOff = int32_t(0x80000000u);

constexpr int kMaxHistory = SMP_MAX_HISTORY;
constexpr int kUnitWords = SMP_MAX_VOCAB / 64 / 32;   // one bit per 64 ids

struct PrepArgs {
  const uint32_t* allowed;   // [batch, words] allowed-token bits, or nullptr
  int words;                 // ceil(vocab / 32)
  const int32_t* history;    // [batch, hist_len] recent token ids, or nullptr
  int hist_len;
  const float* penalty;      // [batch] factors r, or nullptr (no penalty)
};

struct SampleArgs {
  const void* logits;
  int batch;
  int vocab;
  const smp_row_params* params;
  uint64_t seed;
  uint64_t offset;
  int32_t* out_ids;
  float* out_probs;
  int32_t* status;
  float* full_probs;   // debug: [B, V] p~ or NULL
  int32_t* kept;       // debug: [B] |S| or NULL
  PrepArgs prep;       // logit pre-pass (the kernel instance with kPrep only)
  uint64_t row_base;   // global index of row 0 (the Philox counter uses row_base + row)
  uint64_t wait_limit_ns;   // time limit of one wait for a TMA batch
};

// Candidate path: greedy, or valid knobs without top-p and with min-p or a small top-k.
__device__ __forceinline__ bool row_is_fast(const smp_row_params& p, int V) {
  if (row_is_greedy(p)) return true;
  if (!sampling_params_valid(p)) return false;
  if (p.top_p < 1.0f) return false;
  const bool minp = p.min_p > 0.0f && p.min_p < 1.0f;
  const bool topk = p.top_k > 0 && p.top_k < V;
  return minp || (topk && p.top_k <= kFastTopK);
}

// Lower bound, in logits, of {z : exp((z - m) / T) >= min_p} for a row maximum
// of at least m: m + T ln(min_p), lowered by a margin that covers the float
// rounding of the expression.
// The bound is increasing in m, so a running maximum gives a lower bound of
// the final one.  w = T ln(min_p), computed once per row.
__device__ __forceinline__ float minp_bound_w(float m, float w) {
  const float t = m + w;
  return t - (fabsf(m) + fabsf(w)) * 0x1p-20f - 0x1p-126f;
}

// ------------------------------------------------------------------ slices and TMA

// ------------------------------------------------------------------ vector passes



__device__ __forceinline__ void write_error_row(const SampleArgs& a, int b, int flags) {
  a.out_ids[b] = -1;
  if (a.out_probs) a.out_probs[b] = __int_as_float(0x7FC00000);
  if (a.kept) a.kept[b] = 0;
  if (a.status) atomicOr(a.status, flags);
}

// ------------------------------------------------------------------ general path

#include "general.cuh"
#include "general_bf16.cuh"

// ------------------------------------------------------------------ logit pre-pass
//
// Repetition penalty ("Choosing the next word", section "The repetition
// penalty": z_i <- z_i / r for z_i > 0, else z_i * r, for each distinct token
// i among the row's recent tokens) and constraint mask ("Decoding &
// Speculative Sampling", section 39.3: tokens outside the allowed set get
// -inf), applied to every logit the kernel instance with kPrep reads: the
// streamed vectors, the segments read again, the row's edges and the general
// path's passes.  The penalised value is computed in binary32 and kept in the
// logits' precision.

// A row's distinct history ids, sorted, and one bit per unit of 64 ids that
// holds one of them (most ids skip the search on that bit).
struct __align__(16) PrepShared {
  int32_t raw[kMaxHistory];
  int32_t first[kMaxHistory];   // 1 at the first occurrence of a valid id
  int32_t ids[kMaxHistory];
  uint32_t unit_bits[kUnitWords];
  int n;
};

// Nearest bf16 value of a binary32 number (ties to even); NaN and infinities kept.
__device__ __forceinline__ float round_to_bf16(float x) {
  uint32_t b = __float_as_uint(x);
  if ((b & 0x7FFFFFFFu) > 0x7F800000u) return x;
  b = (b + 0x7FFFu + ((b >> 16) & 1u)) & 0xFFFF0000u;
  return __uint_as_float(b);
}

template <typename T>
struct LogitPrep {
  const uint32_t* allowed;   // this row's mask words, or nullptr
  const PrepShared* ps;
  float r;
  __device__ __forceinline__ float operator()(int id, float z) const {
    if (allowed && !((__ldg(allowed + (id >> 5)) >> (id & 31)) & 1u)) return -INFINITY;
    if ((ps->unit_bits[id >> 11] >> ((id >> 6) & 31)) & 1u) {
      int lo = 0, hi = ps->n - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (ps->ids[mid] < id) lo = mid + 1;
        else hi = mid;
      }
      if (ps->ids[lo] == id) {
        z = z > 0.0f ? __fdiv_rn(z, r) : __fmul_rn(z, r);
        if (sizeof(T) == 2) z = round_to_bf16(z);
      }
    }
    return z;
  }
};

__device__ __forceinline__ bool penalty_ok(const SampleArgs& a, int row) {
  if (a.prep.penalty == nullptr) return true;
  const float r = a.prep.penalty[row];
  return isfinite(r) && r > 0.0f;
}

// Whether the 64-id block holding `id` (id < V) holds a history id.
__device__ __forceinline__ bool hist_block(const PrepShared& ps, uint32_t id) {
  return (ps.unit_bits[id >> 11] >> ((id >> 6) & 31)) & 1u;
}

// The allowed bits of the 32 ids from `id` (bit q: id + q), id < V; bits
// past the mask's last word count as allowed.
__device__ __forceinline__ uint32_t allowed_bits32(const uint32_t* w, int words, uint32_t id) {
  if (w == nullptr) return 0xFFFFFFFFu;
  const uint32_t k = id >> 5, sft = id & 31;
  const uint64_t lo = __ldg(w + k);
  const uint64_t hi = int(k) + 1 < words ? __ldg(w + k + 1) : 0xFFFFFFFFull;
  return uint32_t(((hi << 32) | lo) >> sft);
}

// The pre-pass state of a lane's unit (kVecPerLane vectors from token uid0):
// its mask bits and whether its ids may hold a history id.
struct UnitPrep {
  uint32_t w0, w1;   // allowed bits of ids uid0 .. +31 and +32 .. +63
  bool hist;
};

template <typename T>
__device__ __forceinline__ UnitPrep unit_prep(const uint32_t* mrow, int words, int V, uint32_t uid0,
                                              const PrepShared& ps) {
  constexpr int kIds = kVecPerLane * VecOps<T>::kPer;   // 32 (fp32) or 64 (bf16)
  UnitPrep u;
  u.w0 = allowed_bits32(mrow, words, uid0);
  u.w1 = (kIds > 32 && int(uid0) + 32 < V) ? allowed_bits32(mrow, words, uid0 + 32) : 0xFFFFFFFFu;
  u.hist = ps.n > 0 && (hist_block(ps, uid0) || hist_block(ps, uint32_t(min(int(uid0) + kIds - 1, V - 1))));
  return u;
}

// Mask bits of vector jj (0 .. kVecPerLane-1) of a unit.
template <typename T>
__device__ __forceinline__ uint32_t unit_bits_of(const UnitPrep& u, int jj) {
  constexpr int kPer = VecOps<T>::kPer;
  const int off = jj * kPer;
  return off < 32 ? (u.w0 >> off) : (u.w1 >> (off - 32));
}

__device__ __forceinline__ PrepShared& prep_shared();

// First index of the sorted history ids at or past `id`.
__device__ __forceinline__ int hist_lower_bound(const PrepShared& ps, int id) {
  int lo = 0, hi = ps.n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (ps.ids[mid] < id) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// The constraint mask on one vector: each 32-bit word becomes
// (word & keep) | (-inf & ~keep), keep expanding the vector's mask bits
// (bit q: element q allowed) to its elements.
template <typename T>
__device__ __forceinline__ uint4 mask_vec(const uint4& x, uint32_t bits) {
  uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t keep;
    if (sizeof(T) == 2)
      keep = (((bits >> (2 * k)) & 1u) ? 0x0000FFFFu : 0u) | (((bits >> (2 * k + 1)) & 1u) ? 0xFFFF0000u : 0u);
    else
      keep = ((bits >> k) & 1u) ? 0xFFFFFFFFu : 0u;
    const uint32_t ninf = sizeof(T) == 2 ? 0xFF80FF80u : 0xFF800000u;
    w[k] = (w[k] & keep) | (ninf & ~keep);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The mask on a unit held in registers (its first nv vectors).
template <typename T>
__device__ __forceinline__ void mask_regs(uint4 (&xv)[kVecPerLane], int nv, uint32_t w0, uint32_t w1) {
  constexpr uint32_t kFull = (1u << VecOps<T>::kPer) - 1u;
  const UnitPrep up{w0, w1, false};
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j) {
    const uint32_t bits = unit_bits_of<T>(up, j) & kFull;
    if (j < nv && bits != kFull) xv[j] = mask_vec<T>(xv[j], bits);
  }
}

// The repetition penalty (a history id of the unit) and then the mask on a
// unit held in registers: element q of vector j is id uid0 + j kPer + q.
// The history ids inside the unit come from two binary searches; each of
// them is applied by a compare with every element (units with history ids
// are few).
template <typename T>
__device__ __forceinline__ void prep_regs(uint4 (&xv)[kVecPerLane], int nv, uint32_t uid0, uint32_t w0, uint32_t w1,
                                          float r) {
  using Vo = VecOps<T>;
  constexpr int kPer = Vo::kPer;
  const PrepShared& ps = prep_shared();
  const int h0 = hist_lower_bound(ps, int(uid0));
  const int h1 = hist_lower_bound(ps, int(uid0) + nv * kPer);
  for (int t = h0; t < h1; ++t) {
    const int o = ps.ids[t] - int(uid0);
    const int jo = o / kPer, q = o % kPer;
    // element q of a vector: word q / (kPer / 4), half (bf16) q % 2
    const int wi = sizeof(T) == 2 ? (q >> 1) : q;
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j)
      if (j == jo) {
        uint32_t w[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
        const uint32_t word = wi == 0 ? w[0] : wi == 1 ? w[1] : wi == 2 ? w[2] : w[3];
        float z = sizeof(T) == 2 ? __uint_as_float((q & 1) ? (word & 0xFFFF0000u) : (word << 16)) : __uint_as_float(word);
        z = z > 0.0f ? __fdiv_rn(z, r) : __fmul_rn(z, r);
        uint32_t nw;
        if (sizeof(T) == 2) {
          const uint32_t hb = __float_as_uint(round_to_bf16(z)) >> 16;
          nw = (q & 1) ? ((word & 0x0000FFFFu) | (hb << 16)) : ((word & 0xFFFF0000u) | hb);
        } else {
          nw = __float_as_uint(z);
        }
        xv[j] = make_uint4(wi == 0 ? nw : w[0], wi == 1 ? nw : w[1], wi == 2 ? nw : w[2], wi == 3 ? nw : w[3]);
      }
  }
  if ((w0 & w1) != 0xFFFFFFFFu) mask_regs<T>(xv, nv, w0, w1);
}


// Builds the row's PrepShared (history ids in [0, V), each once, sorted).
__device__ __forceinline__ PrepShared& prep_shared() {
  __shared__ PrepShared ps;
  return ps;
}

__device__ __forceinline__ void build_prep(PrepShared& ps, const PrepArgs& pa, int row, int V, bool penalised) {
  const int tid = threadIdx.x;
  const int H = penalised && pa.history ? pa.hist_len : 0;
  for (int w = tid; w < kUnitWords; w += kThreads) ps.unit_bits[w] = 0;
  if (tid < kMaxHistory) {
    int32_t id = -1;
    if (tid < H) id = pa.history[size_t(row) * H + tid];
    ps.raw[tid] = (id >= 0 && id < V) ? id : -1;
  }
  if (tid == 0) ps.n = 0;
  cta_sync();
  // (the loops below read the 64 entries four at a time, every load issued
  // at once)
  const int4* raw4 = reinterpret_cast<const int4*>(ps.raw);
  if (tid < kMaxHistory) {   // first occurrences
    const int32_t id = ps.raw[tid];
    bool first = id >= 0;
#pragma unroll
    for (int s = 0; s < kMaxHistory / 4; ++s) {
      const int4 q = raw4[s];
      first &= !((4 * s < tid && q.x == id) || (4 * s + 1 < tid && q.y == id) ||
                 (4 * s + 2 < tid && q.z == id) || (4 * s + 3 < tid && q.w == id));
    }
    ps.first[tid] = first;
  }
  cta_sync();
  if (tid < kMaxHistory && ps.first[tid]) {   // rank among the distinct ids
    const int32_t id = ps.raw[tid];
    const int4* first4 = reinterpret_cast<const int4*>(ps.first);
    int rank = 0;
#pragma unroll
    for (int s = 0; s < kMaxHistory / 4; ++s) {
      const int4 q = raw4[s], f = first4[s];
      rank += (f.x && q.x < id) + (f.y && q.y < id) + (f.z && q.z < id) + (f.w && q.w < id);
    }
    ps.ids[rank] = id;
    atomicOr(&ps.unit_bits[id >> 11], 1u << ((id >> 6) & 31));
    atomicAdd(&ps.n, 1);
  }
  cta_sync();
}


// ------------------------------------------------------------------ candidate path

struct StreamShared {
  uint64_t full[kBufs];       // TMA completion of each batch buffer
  int timeout;                // a wait ran out of time
  uint32_t cand_n;            // candidates appended for the current row (> kCandMax: overflow)
  uint32_t fin_n;             // candidates at or above the final threshold
  uint32_t maxkey;            // running row maximum as an order key
  unsigned long long zsum;    // Z_S in fixed point
  uint64_t u53;               // the row's uniform (53-bit integer) for the draw
  float c_hi, c_lo;           // log2(e) / T of the row, head and tail
  float w_minp;               // T ln(min_p) of the row (min-p rows)
  uint32_t qn;                // segments to read again
  uint32_t handoffs;          // rows of this CTA marked for the general path
  float red[kWarps];
  uint32_t redu[kWarps];
  uint64_t red64[kWarps];
  uint32_t bc[2];
};

// Candidate lists of a candidate-path row.
struct CandShared {
  float seg[kSegs][kThreads];   // per-lane segment maxima of the row being streamed
  uint32_t q[kThreads];         // segments to read again: lane | segment << 8
  uint32_t hist[256];
  uint32_t cand_id[kCandMax];
  float cand_val[kCandMax];
  uint32_t f_id[kFinalMax];
  float f_val[kFinalMax];
  // The ranked candidates, padded to whole 128-bit loads: (key << 32 | ~id),
  // whose order is the kept-set order, and (id, E_i) with E_i = 0 outside S.
  __align__(16) unsigned long long pk[kFinalMax + 8];
  __align__(16) ulonglong2 idm[kFinalMax + 8];
};

// The general path runs after the CTA's last streamed batch has been
// consumed, so its state lives in the (then idle) batch ring.
static_assert(sizeof(GenShared) <= size_t(kBufs) * kBufBytes, "general-path state must fit the ring");

// Byte layout of a row: the 16-byte aligned middle [a0, a1) streams through
// shared memory in batches of kBufBytes; the few elements before and after it
// are read directly.
struct RowGeom {
  const char* r0;      // first byte of the row
  uintptr_t a0, a1;    // aligned middle (a1 <= a0: no middle)
  int nchunks;         // batches of kBufBytes
  int head;            // elements before a0
  int tail0;           // first element after a1
};

template <typename T>
__device__ __forceinline__ RowGeom row_geom(const SampleArgs& a, int row) {
  RowGeom g;
  g.r0 = reinterpret_cast<const char*>(a.logits) + size_t(row) * a.vocab * sizeof(T);
  const uintptr_t r0 = reinterpret_cast<uintptr_t>(g.r0);
  const uintptr_t r1 = r0 + size_t(a.vocab) * sizeof(T);
  g.a0 = (r0 + 15) & ~uintptr_t(15);
  g.a1 = r1 & ~uintptr_t(15);
  if (g.a1 > g.a0) {
    g.nchunks = int((g.a1 - g.a0 + kBufBytes - 1) / kBufBytes);
    g.head = int((g.a0 - r0) / sizeof(T));
    g.tail0 = int((g.a1 - r0) / sizeof(T));
  } else {
    g.nchunks = 0;
    g.head = a.vocab;
    g.tail0 = a.vocab;
  }
  return g;
}


__device__ __forceinline__ void push_candidate(StreamShared& ss, CandShared& cs, uint32_t id, float z) {
  const uint32_t slot = atomicAdd(&ss.cand_n, 1u);
  if (slot < uint32_t(kCandMax)) {
    cs.cand_id[slot] = id;
    cs.cand_val[slot] = z;
  }
}

// Slots for n entries of this lane in a list counted by *counter, for every
// lane of a converged warp: one atomic per warp.  Returns the lane's first slot.
__device__ __forceinline__ uint32_t warp_reserve(uint32_t* counter, uint32_t n) {
  const uint32_t incl = warp_inclusive_scan<uint32_t>(n);
  uint32_t base = 0;
  if ((threadIdx.x & 31) == 31 && incl) base = atomicAdd(counter, incl);   // lane 31 holds the total
  base = __shfl_sync(0xFFFFFFFFu, base, 31);
  return base + incl - n;
}

// The candidates of one unit held in registers (its first nv vectors, token
// ids from id_first on): every element >= theta, found through a bit mask per
// vector and pushed by a short loop over the set bits.  The row end runs this
// once per row, so its code is kept small.
template <typename T>
__device__ __forceinline__ void push_unit(StreamShared& ss, CandShared& cs, const uint4 (&xv)[kVecPerLane], int nv,
                                          uint32_t id_first, float theta) {
  using V = VecOps<T>;
  constexpr int kPer = V::kPer;
  static_assert(kVecPerLane * kPer <= 64, "one 64-bit mask per unit");
  const uint32_t t = V::threshold(theta);
  unsigned long long m = 0;
#pragma unroll
  for (int j = 0; j < kVecPerLane; ++j)
    if (j < nv) m |= (unsigned long long)V::ge_mask(xv[j], t) << (j * kPer);
#pragma unroll 1
  while (m) {
    const int p = __ffsll((long long)m) - 1;
    m &= m - 1ull;
    const int j = p / kPer, q = p % kPer;
    uint4 x = xv[0];
#pragma unroll
    for (int jj = 1; jj < kVecPerLane; ++jj)
      if (j == jj) x = xv[jj];
    push_candidate(ss, cs, id_first + uint32_t(p), V::elem(x, q));
  }
}

// Exact selection and draw of a min-p / top-k candidate-path row.  The
// candidates hold every element at or above a lower bound of the kept set's
// boundary; row_max is the row's largest logit.  Returns false if the row
// needs the general path.
template <typename T, bool kPrep>
__device__ bool finalize_candidates(StreamShared& ss, CandShared& cs, const FloatPair* table, const SampleArgs& a, int b,
                                    const smp_row_params& prm, float row_max) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int V = a.vocab;
  const bool minp = prm.min_p > 0.0f && prm.min_p < 1.0f;
  const bool topk = prm.top_k > 0 && prm.top_k < V;
  if (!isfinite(row_max)) {
    if (tid == 0) write_error_row(a, b, kRowNonFinite);
    if (a.full_probs)
      for (int i = tid; i < V; i += kThreads) a.full_probs[size_t(b) * V + i] = __int_as_float(0x7FC00000);
    return true;
  }
  if (ss.cand_n > uint32_t(kCandMax)) return false;
  int n = int(ss.cand_n);
  const float* vals = cs.cand_val;
  const uint32_t* ids = cs.cand_id;
  if (n > kFinalMax) {
    // Too many to rank one per thread: keep those at or above the k-th largest value.
    if (!topk || n < prm.top_k) return false;
    float theta = kth_largest_list<T>(cs.cand_val, n, prm.top_k, cs.hist, ss.bc);
    if (minp) theta = fmaxf(theta, minp_bound_w(row_max, ss.w_minp));
    if (tid == 0) ss.fin_n = 0;
    cta_sync();
    for (int i = tid; i < n; i += kThreads) {
      if (!(cs.cand_val[i] >= theta)) continue;
      const uint32_t slot = atomicAdd(&ss.fin_n, 1u);
      if (slot < uint32_t(kFinalMax)) {
        cs.f_id[slot] = cs.cand_id[i];
        cs.f_val[slot] = cs.cand_val[i];
      }
    }
    cta_sync();
    if (ss.fin_n > uint32_t(kFinalMax)) return false;
    n = int(ss.fin_n);
    vals = cs.f_val;
    ids = cs.f_id;
  }
  // Fewer candidates than k: some of the top k are NaN (ranked as -inf).
  // With the pre-pass the candidates exclude -inf (masked tokens), so fewer
  // than k means every finite token is a candidate, and the rest of the top
  // k have zero mass: the candidates decide the draw alone.
  if (!kPrep && topk && n < prm.top_k) return false;

  // Membership of the kept set S, one candidate per thread.
  const bool have = tid < n;
  const float z = have ? vals[tid] : -INFINITY;
  const uint32_t id = have ? ids[tid] : 0xFFFFFFFFu;
  const int n8 = (n + 7) & ~7;
  if (tid < n8) cs.pk[tid] = have ? (uint64_t(key_of_bits(__float_as_uint(z))) << 32) | uint64_t(~id) : 0ull;
  if (topk) cta_sync();
  bool keep = have;
  if (topk && have) {
    // Rank in the order (logit descending, id ascending): the number of
    // larger packed keys.  Every element ranked above a candidate is a
    // candidate, so this is its rank in the row.
    const unsigned long long me = cs.pk[tid];
    const ulonglong2* p2 = reinterpret_cast<const ulonglong2*>(cs.pk);
    int c[4] = {0, 0, 0, 0};
    for (int j = 0; j < n8 / 2; j += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const ulonglong2 q = p2[j + u];
        c[u] += int(q.x > me) + int(q.y > me);
      }
    }
    keep = c[0] + c[1] + c[2] + c[3] < prm.top_k;
  }
  // One exponential per candidate gives both the exact min-p test and the mass.
  RowScale rs;
  rs.m = row_max;
  rs.c_hi = ss.c_hi;
  rs.c_lo = ss.c_lo;
  uint64_t e = 0;
  if (keep) {
    const ExpParts p = exp_parts(z, rs, table, -1000.0f);
    if (minp) keep = parts_at_least(p, prm.min_p);
    if (keep) e = fixed_from_parts(p);
  }
  if (tid < n8) cs.idm[tid] = make_ulonglong2(have ? id : 0xFFFFFFFFull, e);
  const uint64_t ws = warp_sum<uint64_t>(e);
  if (lane == 0 && ws) atomicAdd(&ss.zsum, (unsigned long long)ws);
  const int kept = cta_sync_count(keep);
  const uint64_t z_kept = ss.zsum;
  // The draw: the kept token (id order) whose cumulative mass interval holds
  // t = floor(u * Z_S), u = Philox draw 0 of row b.
  const uint64_t t = uint64_t((u128(ss.u53) * z_kept) >> 53);
  if (keep && e) {
    uint64_t c[4] = {0, 0, 0, 0};
    for (int j = 0; j < n8; j += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const ulonglong2 q = cs.idm[j + u];
        c[u] += q.x < id ? q.y : 0ull;
      }
    }
    const uint64_t before = c[0] + c[1] + c[2] + c[3];
    if (before <= t && t - before < e) {
      a.out_ids[b] = int32_t(id);
      if (a.out_probs) a.out_probs[b] = __fdividef(float(e), float(z_kept));   // within 2 ulp
    }
  }
  if (tid == 0 && a.kept) a.kept[b] = kept;
  if (a.full_probs) {
    for (int i = tid; i < V; i += kThreads) a.full_probs[size_t(b) * V + i] = 0.0f;
    cta_sync();
    if (keep && e) a.full_probs[size_t(b) * V + id] = __fdiv_rn(float(e), float(z_kept));
  }
  return true;
}

// ------------------------------------------------------------------ the kernel
//
// One CTA per row (CTA i takes rows i, i + grid, ...).  A candidate-path row
// streams through two kBufBytes buffers in shared memory, each filled by one
// TMA bulk copy; thread 0 refills a buffer as soon as the CTA is done with it,
// running ahead across row boundaries.  The first batches of a CTA's first row
// are requested before the row's knobs are read.  Each warp takes one
// kSubBytes part of a batch; each lane one unit of kVecPerLane consecutive
// 16-byte vectors (a 128-byte line, so that a unit read again from global
// memory is one line).
//   greedy:  every lane keeps its (max, lowest id) in registers; one CTA-wide
//            arg-max at the end of the row.
//   min-p:   candidates are the elements >= running maximum + T ln(min_p)
//            (lowered by a rounding margin); the running maximum is shared
//            through an atomicMax on order keys.
//   top-k:   candidates are the elements >= the k-th largest per-lane
//            maximum of the first batch, raised to the k-th largest candidate
//            when the list is compacted.
// A warp gathers its candidates of a batch in a per-lane bit mask and appends
// them with one atomic.  Every threshold is a lower bound of the kept set's
// boundary, so the candidates contain the kept set; the end of the row selects
// it exactly.  General-path rows, and rows whose candidates overflow, are
// marked (out_ids = kHandOff) and taken by the general path once the CTA's
// candidate-path rows are done, so that none of its state is live across it.

// Cursor over the batches of this CTA's candidate-path rows (thread 0 only).
template <typename T, bool kPrep>
struct BatchCursor {
  int row;
  int batch;
  int nbatch;
  uint32_t issued;   // copies requested so far
  uint64_t policy;   // L2 policy of the copies

  // Start at this CTA's first row before its knobs are known.
  __device__ void begin(const SampleArgs& a) {
    row = blockIdx.x;
    batch = 0;
    nbatch = row < a.batch ? row_geom<T>(a, row).nchunks : 0;
    issued = 0;
    policy = evict_first_policy();
  }
  // The first row's knobs are known: a general-path row stops after the
  // batches already requested.  When the ring is deeper than that row, the
  // cursor has moved on to later rows, whose knobs it read: nothing to stop.
  __device__ void known(bool fast) {
    if (!fast && row == int(blockIdx.x)) nbatch = batch;
  }
  __device__ void settle(const SampleArgs& a) {
    while (row < a.batch && batch >= nbatch) {
      row += gridDim.x;
      batch = 0;
      nbatch = 0;
      if (row < a.batch) {
        const smp_row_params prm = a.params[row];
        const bool fast = row_is_fast(prm, a.vocab) && (!kPrep || penalty_ok(a, row));
        nbatch = fast ? row_geom<T>(a, row).nchunks : 0;
      }
    }
  }
  __device__ void issue(const SampleArgs& a, unsigned char* dst, uint64_t* bar) {
    settle(a);
    if (row >= a.batch) return;
    const RowGeom g = row_geom<T>(a, row);
    const uintptr_t src = g.a0 + uintptr_t(batch) * kBufBytes;
    const uint32_t bytes = uint32_t(min(uintptr_t(kBufBytes), g.a1 - src));
    tma_load(dst, reinterpret_cast<const void*>(src), bytes, bar, policy);
    ++batch;
    ++issued;
  }
};

// kPrep: the instance of smp_sample_processed, which applies the logit
// pre-pass to every value it reads; without it the kernel carries none of
// that code.
template <typename T, bool kPrep>
__global__ void __launch_bounds__(kThreads, 2) sample_kernel(SampleArgs a) {
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ StreamShared ss;
  __shared__ FloatPair table[64];
  __shared__ CandShared cs;
  using V = VecOps<T>;
  constexpr int kPer = V::kPer;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int B = a.batch;
  const int Vn = a.vocab;
  BatchCursor<T, kPrep> cur;
  if (tid == 0) {
    for (int i = 0; i < kBufs; ++i) mbar_init(&ss.full[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // The first batches of the CTA's first row are prefetched into L2 before
  // the dependency wait: a prefetch is a hint that changes no memory, and L2
  // is the point of coherence, so writes the previous kernel makes to these
  // bytes still reach the copies below.  In a chain of launches the prefetch
  // overlaps the previous launch's row ends, when HBM is otherwise idle.
  if (tid == 0 && int(blockIdx.x) < B) {
    const RowGeom g = row_geom<T>(a, blockIdx.x);
    const int nb = min(g.nchunks, kPrefetchBatches);
    for (int bt = 0; bt < nb; ++bt) {
      const uintptr_t src = g.a0 + uintptr_t(bt) * kBufBytes;
      const uint32_t bytes = uint32_t(min(uintptr_t(kBufBytes), g.a1 - src));
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
    }
  }
  // Inputs may come from the previous kernel on the stream (programmatic launch).
  grid_dependency_wait();
  if (tid == 0) {
    cur.begin(a);
    for (int i = 0; i < kBufs; ++i) cur.issue(a, ring + size_t(i) * kBufBytes, &ss.full[i]);
    ss.timeout = 0;
    ss.handoffs = 0;
  }
  allow_dependent_launch();
  if (tid < 64) table[tid] = kExp2Table[tid];
  cta_sync();

  uint32_t consumed = 0;   // batches consumed so far (the buffers' running index)
  bool alive = true;
  int row = blockIdx.x;   // after the loop: the row a wait ran out of time on
  for (; row < B && alive; row += gridDim.x) {
    const smp_row_params prm = a.params[row];
    const RowGeom geo = row_geom<T>(a, row);
    const bool first = row == int(blockIdx.x);
    const bool fast = row_is_fast(prm, Vn) && (!kPrep || penalty_ok(a, row));
    const T* rowp = reinterpret_cast<const T*>(geo.r0);
    if (!fast) {
      if (first && geo.nchunks > 0) {
        // Let the speculative copies land and hand their buffers to the next rows.
        const int spec = min(kBufs, geo.nchunks);
        if (tid == 0) {
          cur.known(false);
          for (int s = 0; s < spec; ++s) {
            const uint32_t k = consumed + uint32_t(s);
            if (!wait_full(&ss.full[k % kBufs], (k / kBufs) & 1, a.wait_limit_ns)) {
              ss.timeout = 1;
              break;
            }
            cur.issue(a, ring + size_t(k % kBufs) * kBufBytes, &ss.full[k % kBufs]);
          }
        }
        cta_sync();
        if (ss.timeout) {
          alive = false;
          break;
        }
        consumed += uint32_t(spec);
      }
      if (tid == 0) {
        a.out_ids[row] = kHandOff;
        ++ss.handoffs;
      }
      continue;
    }
    const bool greedy = row_is_greedy(prm);
    const bool minp = !greedy && prm.min_p > 0.0f && prm.min_p < 1.0f;
    const bool topk = !greedy && prm.top_k > 0 && prm.top_k < Vn;
    if (tid == 0) {
      ss.cand_n = 0;
      ss.maxkey = 0;
    }
    if (!greedy && tid == kThreads - 1) {
      // Row constants of the draw, off the critical path of the stream.
      ss.u53 = uniform53(a.seed, a.offset, a.row_base + uint64_t(row), 0);
      const RowScale r0 = make_row_scale(0.0f, prm.temperature);
      ss.c_hi = r0.c_hi;
      ss.c_lo = r0.c_lo;
      ss.w_minp = minp ? prm.temperature * logf(prm.min_p) : 0.0f;
      ss.zsum = 0;
    }
    cta_sync();
    // The row's pre-pass state (kPrep): its mask words, its distinct history
    // ids and its factor; xf applies the pre-pass to one element.
    const uint32_t* mrow = nullptr;
    float prep_r = 1.0f;
    if constexpr (kPrep) {
      mrow = a.prep.allowed ? a.prep.allowed + size_t(row) * a.prep.words : nullptr;
      prep_r = a.prep.penalty ? a.prep.penalty[row] : 1.0f;
      build_prep(prep_shared(), a.prep, row, Vn, prep_r != 1.0f);
    }
    auto xf = [&](uint32_t id, float z) -> float {
      if constexpr (kPrep) return LogitPrep<T>{mrow, &prep_shared(), prep_r}(int(id), z);
      return z;
    };
    const uint32_t id_base = uint32_t((geo.a0 - reinterpret_cast<uintptr_t>(geo.r0)) / sizeof(T));
    const int v0 = warp * (kSubBytes / 16);            // this warp's first vector in every batch
    const int seg_len = (geo.nchunks + kSegs - 1) / kSegs;   // batches per segment
    float best_z = -INFINITY;      // greedy: this lane's maximum and its lowest id
    uint32_t best_id = 0xFFFFFFFFu;
    float seg_max = -INFINITY;     // other rows: this lane's maximum over the current segment
    float lane_row_max = -INFINITY;   // ... and over the row
    // The raw mask words of this lane's unit in batch bt2 (the fused
    // pre-pass with a mask), combined when the batch is processed.
    struct MaskRaw {
      uint32_t a, b, c, sft;
      bool on, w1;
    };
    auto mask_load = [&](int bt2) -> MaskRaw {
      MaskRaw m{0xFFFFFFFFu, 0xFFFFFFFFu, 0xFFFFFFFFu, 0u, false, false};
      if constexpr (kPrep) {
        const uintptr_t bst = geo.a0 + uintptr_t(bt2) * kBufBytes;
        const int bv = int(min(uintptr_t(kBufBytes), geo.a1 - bst) / 16);
        const int nv2 = max(0, min(bv - v0, kSubBytes / 16));
        if (mrow && lane * kVecPerLane < nv2) {
          const uint32_t uid0 = id_base + uint32_t(bt2) * (kBufBytes / sizeof(T)) + uint32_t(v0 * kPer) +
                                uint32_t(lane * kVecPerLane * kPer);
          const uint32_t k = uid0 >> 5;
          const int words = a.prep.words;
          m.on = true;
          m.sft = uid0 & 31u;
          m.w1 = kVecPerLane * kPer > 32 && int(uid0) + 32 < Vn;
          m.a = __ldg(mrow + k);
          m.b = int(k) + 1 < words ? __ldg(mrow + k + 1) : 0xFFFFFFFFu;
          m.c = m.w1 && int(k) + 2 < words ? __ldg(mrow + k + 2) : 0xFFFFFFFFu;
        }
      }
      return m;
    };
    MaskRaw mnext = mask_load(0);

    for (int bt = 0; bt < geo.nchunks; ++bt) {
      const uint32_t bi = consumed % kBufs;
      // This warp's part of the batch.
      const uintptr_t bstart = geo.a0 + uintptr_t(bt) * kBufBytes;
      const int bvec = int(min(uintptr_t(kBufBytes), geo.a1 - bstart) / 16);
      const int nvec = max(0, min(bvec - v0, kSubBytes / 16));
      const uint4* vec = reinterpret_cast<const uint4*>(ring + size_t(bi) * kBufBytes) + v0;
      const T* part = reinterpret_cast<const T*>(vec);
      const uint32_t id0 = id_base + uint32_t(bt) * (kBufBytes / sizeof(T)) + uint32_t(v0 * kPer);
      // The mask bits of the lane's unit: its words were requested one batch
      // ahead (and the next batch's are requested now), so that their latency
      // overlaps a whole batch.
      uint32_t mw0 = 0xFFFFFFFFu, mw1 = 0xFFFFFFFFu;
      if constexpr (kPrep) {
        if (mnext.on) {
          mw0 = uint32_t(((uint64_t(mnext.b) << 32) | mnext.a) >> mnext.sft);
          if (mnext.w1) mw1 = uint32_t(((uint64_t(mnext.c) << 32) | mnext.b) >> mnext.sft);
        }
        if (bt + 1 < geo.nchunks) mnext = mask_load(bt + 1);
      }
      if (!wait_full(&ss.full[bi], (consumed / kBufs) & 1, a.wait_limit_ns)) ss.timeout = 1;
      // The lane's batch maximum: one packed maximum over its unit, the
      // kVecPerLane consecutive vectors (one 128-byte line) from lane *
      // kVecPerLane, read in the order j ^ (lane % 8) so that the 32 lanes of
      // a step touch all banks evenly.
      uint32_t pm = V::neg_inf();
      if constexpr (kPrep) {
        const PrepShared& ps = prep_shared();
        if (ps.n > 0) {
          // The penalty, in place in the ring: thread t takes history id t if
          // it lies in this batch; one barrier before the lanes read.
          if (tid < ps.n) {
            const uint32_t bid0 = id_base + uint32_t(bt) * (kBufBytes / sizeof(T));
            const uint32_t e = uint32_t(ps.ids[tid]) - bid0;
            if (uint32_t(ps.ids[tid]) >= bid0 && e < uint32_t(bvec) * uint32_t(kPer)) {
              T* slot = reinterpret_cast<T*>(ring + size_t(bi) * kBufBytes) + e;
              float z = Elem<T>::widen(*slot);
              z = z > 0.0f ? __fdiv_rn(z, prep_r) : __fmul_rn(z, prep_r);
              if (sizeof(T) == 2) *reinterpret_cast<uint16_t*>(slot) = uint16_t(__float_as_uint(round_to_bf16(z)) >> 16);
              else *reinterpret_cast<float*>(slot) = z;
            }
          }
          cta_sync();
        }
      }
      // (with a mask: each vector masked in registers as it is read, and
      // written back to the ring when one of its bits is clear)
      bool masking = false;
      if constexpr (kPrep) masking = mrow && (mw0 & mw1) != 0xFFFFFFFFu;
#pragma unroll
      for (int j = 0; j < kVecPerLane; ++j) {
        const int jj = j ^ (lane & (kVecPerLane - 1));
        const int v = lane * kVecPerLane + jj;
        if (v < nvec) {
          uint4 x = vec[v];
          if constexpr (kPrep) {
            const uint32_t bits = unit_bits_of<T>(UnitPrep{mw0, mw1, false}, jj) & ((1u << kPer) - 1u);
            if (masking && bits != (1u << kPer) - 1u) {
              x = mask_vec<T>(x, bits);
              const_cast<uint4*>(vec)[v] = x;
            }
          }
          pm = V::max2(pm, V::vmax(x));
        }
      }
      const float lane_max = V::finish(pm);
      const uint32_t lane_key = lane_max > -INFINITY ? key_of_bits(__float_as_uint(lane_max)) : 0u;
      const uint32_t wkey = __reduce_max_sync(0xFFFFFFFFu, lane_key);
      if (greedy) {
        // Only a lane whose batch maximum beats its own best and reaches the
        // CTA's running maximum can hold the row's arg-max: locate its first
        // occurrence (ids rise with j, then q; the lane's valid vectors come
        // first).
        const uint32_t shared_key = *reinterpret_cast<volatile uint32_t*>(&ss.maxkey);
        const float shared_max = shared_key ? value_of_key(shared_key) : -INFINITY;
        if (lane_max > best_z && lane_max >= shared_max) {
          for (int j = 0; j < kVecPerLane && lane * kVecPerLane + j < nvec; ++j) {
            const int e0 = (lane * kVecPerLane + j) * kPer;
            int hit = -1;
#pragma unroll
            for (int q = kPer - 1; q >= 0; --q)
              if (Elem<T>::widen(part[e0 + q]) == lane_max) hit = q;
            if (hit >= 0) {
              best_id = id0 + uint32_t(e0 + hit);
              break;
            }
          }
          best_z = lane_max;
        }
      } else {
        seg_max = fmaxf(seg_max, lane_max);
        lane_row_max = fmaxf(lane_row_max, lane_max);
        if (bt % seg_len == seg_len - 1 || bt == geo.nchunks - 1) {
          cs.seg[bt / seg_len][tid] = seg_max;
          seg_max = -INFINITY;
        }
      }
      if (lane == 0 && wkey) atomicMax(&ss.maxkey, wkey);
      cta_sync();   // the buffer is free
      if (ss.timeout) {
        // This batch's copy may still be in flight: `consumed` stays on it,
        // so that the clean-up below waits for it too.
        alive = false;
        break;
      }
      ++consumed;
      if (tid == 0) cur.issue(a, ring + size_t(bi) * kBufBytes, &ss.full[bi]);
    }
    if (!alive) break;

    if (greedy) {
      // Elements outside the aligned middle; then the CTA-wide (max, lowest id).
      uint64_t best = pack_key_id(key_of_bits(__float_as_uint(best_z)), best_id);
      for (int i = tid; i < geo.head; i += kThreads) {
        const uint64_t p = pack_key_id(key_of_bits(__float_as_uint(xf(i, Elem<T>::widen(rowp[i])))), uint32_t(i));
        best = p > best ? p : best;
      }
      for (int i = geo.tail0 + tid; i < Vn; i += kThreads) {
        const uint64_t p = pack_key_id(key_of_bits(__float_as_uint(xf(i, Elem<T>::widen(rowp[i])))), uint32_t(i));
        best = p > best ? p : best;
      }
      best = block_max_u64(best, ss.red64);
      const float row_max = value_of_key(uint32_t(best >> 32));
      const uint32_t tok = ~uint32_t(best);
      if (!isfinite(row_max)) {
        if (tid == 0) write_error_row(a, row, kRowNonFinite);
        if (a.full_probs)
          for (int i = tid; i < Vn; i += kThreads) a.full_probs[size_t(row) * Vn + i] = __int_as_float(0x7FC00000);
      } else {
        if (tid == 0) {
          a.out_ids[row] = int32_t(tok);
          if (a.out_probs) a.out_probs[row] = 1.0f;
          if (a.kept) a.kept[row] = 1;
        }
        if (a.full_probs)
          for (int i = tid; i < Vn; i += kThreads)
            a.full_probs[size_t(row) * Vn + i] = uint32_t(i) == tok ? 1.0f : 0.0f;
      }
      cta_sync();
      continue;
    }

    // The row maximum, with the elements outside the aligned middle.
    float run_max = ss.maxkey ? value_of_key(ss.maxkey) : -INFINITY;
    const bool edges = geo.head > 0 || geo.tail0 < Vn;
    if (edges) {
      float emax = -INFINITY;
      for (int i = tid; i < geo.head; i += kThreads) emax = fmaxf(emax, xf(i, Elem<T>::widen(rowp[i])));
      for (int i = geo.tail0 + tid; i < Vn; i += kThreads) emax = fmaxf(emax, xf(i, Elem<T>::widen(rowp[i])));
      run_max = fmaxf(run_max, block_max_f(emax, ss.red));
    }
    // A lower bound theta of the kept set's boundary: min-p's at the row
    // maximum, and the k-th largest per-lane maximum (k lanes hold an element
    // at least that large, so the k-th largest element is too).
    float theta = -INFINITY;
    if (minp) theta = minp_bound_w(run_max, ss.w_minp);
    const int nseg = (geo.nchunks + seg_len - 1) / seg_len;
    if (topk) {
      // Two 8-bit radix levels over the lane maxima (the candidate values are
      // not in use yet).
      cs.cand_val[tid] = lane_row_max;
      cta_sync();
      theta = fmaxf(theta, kth_largest_list<T>(cs.cand_val, kThreads, prm.top_k, cs.hist, ss.bc));
    }
    // With the pre-pass, masked tokens (-inf, zero mass) are never
    // candidates, so that a row with few allowed tokens stays on this path.
    if constexpr (kPrep)
      if (!isnan(theta)) theta = fmaxf(theta, __uint_as_float(0xFF7FFFFFu));   // the lowest finite float
    // Candidates: every element >= theta, from the segments whose maximum
    // reaches it (read again from global memory, normally still in L2) and
    // from the edges.
    if (tid == 0) ss.qn = 0;
    cta_sync();
    if (!isnan(theta)) {
      // The (lane, segment) pairs to read again, then one pass in which every
      // thread takes one of them (all its loads in flight at once).
      // Each lane lists its own pairs; a warp appends them with one atomic.
      uint32_t hits = 0;   // this lane's segments at or above theta (nseg <= kSegs)
      for (int sgi = 0; sgi < nseg; ++sgi) hits |= (cs.seg[sgi][tid] >= theta ? 1u : 0u) << sgi;
      uint32_t slot = warp_reserve(&ss.qn, uint32_t(__popc(hits)));
      while (hits) {
        const int sgi = __ffs(hits) - 1;
        hits &= hits - 1u;
        if (slot < uint32_t(kThreads)) cs.q[slot] = uint32_t(tid) | (uint32_t(sgi) << 8);
        ++slot;
      }
      cta_sync();
      const int qn = int(ss.qn);
      if (qn > kThreads) {
        if (tid == 0) ss.cand_n = uint32_t(kCandMax) + 1;   // too many: the general path takes the row
      } else {
        for (int w = tid; w < qn * seg_len; w += kThreads) {
          const uint32_t pr = cs.q[w / seg_len];
          const int owner = int(pr & 255u);
          const int bt = int(pr >> 8) * seg_len + w % seg_len;
          if (bt >= geo.nchunks) continue;
          const int ov0 = (owner >> 5) * (kSubBytes / 16);
          const int ol = owner & 31;
          const uintptr_t bstart = geo.a0 + uintptr_t(bt) * kBufBytes;
          const int bvec = int(min(uintptr_t(kBufBytes), geo.a1 - bstart) / 16);
          const int nvec = max(0, min(bvec - ov0, kSubBytes / 16));
          const uint4* gv = reinterpret_cast<const uint4*>(bstart) + ov0;
          const uint32_t id0 = id_base + uint32_t(bt) * (kBufBytes / sizeof(T)) + uint32_t(ov0 * kPer);
          uint4 xv[kVecPerLane];   // the owner's unit: one 128-byte line
#pragma unroll
          for (int j = 0; j < kVecPerLane; ++j) {
            const int v = ol * kVecPerLane + j;
            xv[j] = v < nvec ? __ldg(gv + v) : make_uint4(V::neg_inf(), V::neg_inf(), V::neg_inf(), V::neg_inf());
          }
          if constexpr (kPrep) {
            if (ol * kVecPerLane < nvec) {
              const uint32_t uid0 = id0 + uint32_t(ol * kVecPerLane * kPer);
              const UnitPrep up = unit_prep<T>(mrow, a.prep.words, Vn, uid0, prep_shared());
              if (up.hist)
                prep_regs<T>(xv, min(kVecPerLane, nvec - ol * kVecPerLane), uid0, up.w0, up.w1, prep_r);
              else if ((up.w0 & up.w1) != 0xFFFFFFFFu)
                mask_regs<T>(xv, min(kVecPerLane, nvec - ol * kVecPerLane), up.w0, up.w1);
            }
          }
          push_unit<T>(ss, cs, xv, min(kVecPerLane, max(0, nvec - ol * kVecPerLane)),
                       id0 + uint32_t(ol * kVecPerLane * kPer), theta);
        }
      }
      for (int i = tid; i < geo.head; i += kThreads) {
        const float z = xf(i, Elem<T>::widen(rowp[i]));
        if (z >= theta) push_candidate(ss, cs, uint32_t(i), z);
      }
      for (int i = geo.tail0 + tid; i < Vn; i += kThreads) {
        const float z = xf(i, Elem<T>::widen(rowp[i]));
        if (z >= theta) push_candidate(ss, cs, uint32_t(i), z);
      }
    }
    cta_sync();
    if (!finalize_candidates<T, kPrep>(ss, cs, table, a, row, prm, run_max) && tid == 0) {
      a.out_ids[row] = kHandOff;
      ++ss.handoffs;
    }
    cta_sync();
  }
  // Thread 0 marks rows and counts them without a barrier after the last
  // row: every thread must see the same marks and count before it branches.
  cta_sync();
  if (!alive) {
    // A wait ran out of time: let the copies in flight land (with the
    // default limit, whatever the call's: the CTA must not exit while a copy
    // still writes its shared memory), and give the rows from that one on,
    // and the marked rows, the error result.
    if (tid == 0)
      for (uint32_t k = consumed; k < cur.issued; ++k) wait_full(&ss.full[k % kBufs], (k / kBufs) & 1, kWaitLimitNs);
    for (int r = blockIdx.x; r < B; r += gridDim.x) {
      if (r < row && load_volatile(a.out_ids + r) != kHandOff) continue;
      cta_sync();
      if (tid == 0) write_error_row(a, r, kRowTimeout);
      if (a.full_probs)
        for (int i = tid; i < Vn; i += kThreads) a.full_probs[size_t(r) * Vn + i] = __int_as_float(0x7FC00000);
    }
    cta_sync();
    return;
  }
  // The marked rows, by the general path (its state overlays the idle ring).
  if (ss.handoffs == 0) return;
  GenShared& gen = *reinterpret_cast<GenShared*>(ring);
  for (int r = blockIdx.x; r < B; r += gridDim.x) {
    // Every thread reads the mark before the row's first barrier; the row's
    // result replaces it only after later barriers.
    if (load_volatile(a.out_ids + r) != kHandOff) continue;
    const smp_row_params prm = a.params[r];
    if constexpr (kPrep) {
      if (!penalty_ok(a, r)) {   // an invalid factor: an error row (after every thread read the mark)
        cta_sync();
        if (tid == 0) write_error_row(a, r, kRowBadParams);
        continue;
      }
      const float rr = a.prep.penalty ? a.prep.penalty[r] : 1.0f;
      build_prep(prep_shared(), a.prep, r, Vn, rr != 1.0f);
      const uint32_t* mr = a.prep.allowed ? a.prep.allowed + size_t(r) * a.prep.words : nullptr;
      const LogitPrep<T> xf{mr, &prep_shared(), rr};
      bool done = false;
      if constexpr (sizeof(T) == 2) done = key_table_row(*reinterpret_cast<KeyTable*>(ring), table, a, r, prm, xf);
      if (!done) general_row<T>(gen, table, a, r, prm, xf);
    } else {
      bool done = false;
      if constexpr (sizeof(T) == 2) done = key_table_row(*reinterpret_cast<KeyTable*>(ring), table, a, r, prm);
      if (!done) general_row<T>(gen, table, a, r, prm);
    }
  }
}

// ------------------------------------------------------------------ host side

template <typename T, bool kPrep = false>
static smp_status launch_sample(const SampleArgs& args, cudaStream_t stream) {
  const int dev = current_device();
  if (dev < 0) return fail_cuda(cudaGetLastError());
  LaunchShape ls;
  ls.cluster = 1;
  ls.smem = size_t(kBufs) * kBufBytes;
  ls.pdl = true;
  const void* kernel = reinterpret_cast<const void*>(&sample_kernel<T, kPrep>);
  cudaError_t err = prepare_kernel(kernel, dev, ls);
  if (err != cudaSuccess) return fail_cuda(err);
  int per_sm = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, ls.smem);
  if (err != cudaSuccess) return fail_cuda(err);
  if (per_sm <= 0) return SMP_ERR_UNSUPPORTED;
  const int resident = per_sm * device_sms(dev);
  const int grid = args.batch < resident ? args.batch : resident;
  if (verbose())
    fprintf(stderr, "smp_sample: batch %d vocab %d grid %d (%d CTAs/SM) ring %zu bytes\n", args.batch,
            args.vocab, grid, per_sm, ls.smem);
  SampleArgs a = args;
  err = launch_cluster(kernel, dim3(grid), dim3(kThreads), ls, stream, &a);
  if (err != cudaSuccess) return fail_cuda(err);
  return SMP_OK;
}

// Every sampler entry point: argument checks, then the status clear and the
// kernel instance (with the logit pre-pass when any of its inputs is given).
static smp_status sample_entry(const void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                               const smp_row_params* params, const uint32_t* allowed, const int32_t* history,
                               int32_t history_len, const float* penalty, uint64_t seed, uint64_t offset,
                               uint64_t row_base, int32_t* out_ids, float* out_probs, float* full, int32_t* kept,
                               int32_t* status, void* stream) {
  if (dtype != SMP_F32 && dtype != SMP_BF16) return SMP_ERR_DTYPE;
  if (!logits || !params || !out_ids) return SMP_ERR_INVALID_ARG;
  if (batch <= 0 || vocab <= 0) return SMP_ERR_INVALID_ARG;
  if (vocab > SMP_MAX_VOCAB) return SMP_ERR_UNSUPPORTED;
  if (history_len < 0 || history_len > SMP_MAX_HISTORY || (history_len > 0 && !history))
    return SMP_ERR_INVALID_ARG;
  const int elem = dtype == SMP_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(logits) % elem) return SMP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(params) | reinterpret_cast<uintptr_t>(out_ids) |
       reinterpret_cast<uintptr_t>(out_probs) | reinterpret_cast<uintptr_t>(allowed) |
       reinterpret_cast<uintptr_t>(history) | reinterpret_cast<uintptr_t>(penalty) |
       reinterpret_cast<uintptr_t>(full) | reinterpret_cast<uintptr_t>(kept)) % 4)
    return SMP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (status) {
    const smp_status rc = clear_status(status, st);
    if (rc != SMP_OK) return rc;
  }
  SampleArgs a{};
  a.logits = logits;
  a.batch = batch;
  a.vocab = vocab;
  a.params = params;
  a.seed = seed;
  a.offset = offset;
  a.row_base = row_base;
  a.wait_limit_ns = wait_limit_ns();
  a.out_ids = out_ids;
  a.out_probs = out_probs;
  a.status = status;
  a.full_probs = full;
  a.kept = kept;
  a.prep.allowed = allowed;
  a.prep.words = (vocab + 31) / 32;
  a.prep.history = history_len > 0 ? history : nullptr;
  a.prep.hist_len = history_len;
  a.prep.penalty = penalty;
  const bool prep = allowed || history_len > 0 || penalty;
  if (prep) return dtype == SMP_F32 ? launch_sample<float, true>(a, st) : launch_sample<uint16_t, true>(a, st);
  return dtype == SMP_F32 ? launch_sample<float>(a, st) : launch_sample<uint16_t>(a, st);
}

}  // namespace smp

extern "C" smp_status smp_sample(const void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                                 const smp_row_params* params, uint64_t seed, uint64_t offset,
                                 int32_t* out_ids, float* out_probs, int32_t* status, void* stream) {
  return smp::sample_entry(logits, batch, vocab, dtype, params, nullptr, nullptr, 0, nullptr, seed, offset, 0,
                           out_ids, out_probs, nullptr, nullptr, status, stream);
}

extern "C" smp_status smp_filter_debug(const void* logits, int32_t batch, int32_t vocab,
                                       smp_dtype dtype, const smp_row_params* params, uint64_t seed,
                                       uint64_t offset, int32_t* out_ids, float* out_probs,
                                       float* out_probs_full, int32_t* out_kept, int32_t* status,
                                       void* stream) {
  if (!out_probs_full || !out_kept) return SMP_ERR_INVALID_ARG;
  return smp::sample_entry(logits, batch, vocab, dtype, params, nullptr, nullptr, 0, nullptr, seed, offset, 0,
                           out_ids, out_probs, out_probs_full, out_kept, status, stream);
}

extern "C" smp_status smp_sample_processed(const void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                                           const smp_row_params* params, const uint32_t* allowed,
                                           const int32_t* history, int32_t history_len,
                                           const float* repetition_penalty, uint64_t seed, uint64_t offset,
                                           int32_t* out_ids, float* out_probs, int32_t* status, void* stream) {
  return smp::sample_entry(logits, batch, vocab, dtype, params, allowed, history, history_len, repetition_penalty,
                           seed, offset, 0, out_ids, out_probs, nullptr, nullptr, status, stream);
}

extern "C" smp_status smp_sample_rows(const void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                                      const smp_row_params* params, const uint32_t* allowed, const int32_t* history,
                                      int32_t history_len, const float* repetition_penalty, uint64_t seed,
                                      uint64_t offset, uint64_t row_base, int32_t* out_ids, float* out_probs,
                                      int32_t* status, void* stream) {
  return smp::sample_entry(logits, batch, vocab, dtype, params, allowed, history, history_len, repetition_penalty,
                           seed, offset, row_base, out_ids, out_probs, nullptr, nullptr, status, stream);
}
