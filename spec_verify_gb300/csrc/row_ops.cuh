// Row-level operations on a vocabulary slice held in shared memory by each
// CTA of a cluster: loading with the row maximum, cluster exchanges through
// mailboxes, radix selection of the kept-set boundary, and the id-order draw.
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

template <typename T>
__device__ __forceinline__ uint32_t elem_key(T v) {
  const uint32_t k = key_of_bits(Elem<T>::bits(v));
  return KeyTraits<T>::kBits == 32 ? k : (k >> 16);
}

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

// Mailbox: partial results one CTA publishes for its peers.
struct Mailbox {
  uint64_t mass[256];
  uint32_t count[256];
  uint64_t w[8];
  u128 x[2];
};

// Shared state of one CTA while it works on a row.
struct RowShared {
  Mailbox mbox[2];
  uint64_t mbar;
  int ok;
  uint32_t hist_cnt[256];
  uint64_t hist_mass[256];
  uint32_t tot_cnt[256];
  uint64_t tot_mass[256];
  uint32_t rank_cnt[kMaxCluster];
  uint64_t red64[kWarps];
  u128 red128[kWarps];
  uint32_t red32[kWarps];
  uint64_t bcast64[8];
  uint32_t bcast32[8];
};

template <typename T>
struct RowCtx {
  RowShared* sh;
  const FloatPair* table;   // 2^(j/64) table of the exponential, in shared memory
  const T* s;          // slice: element i has global id lo + i
  int n;               // elements in this CTA's slice (may be 0)
  int lo;              // global id of element 0
  uint32_t rank;        // index of this CTA within the group
  uint32_t nranks;      // CTAs working on the row
  uint32_t first;       // cluster rank of member 0 (members are first .. first + nranks - 1)
  ClusterBarrier* cb;  // barrier of the group (its phase state outlives one row)
  int mb;              // mailbox buffer in use
  bool alive;          // false after a timeout

  __device__ Mailbox& mine() { return sh->mbox[mb]; }
  __device__ uint32_t peer_addr(const void* field, uint32_t r) const {
    return map_rank(smem_addr(field), first + r);
  }

  // Publish-then-read: call after writing mine(); returns after the barrier.
  __device__ bool exchange() {
    alive = alive && cb->sync();
    return alive;
  }
  __device__ void flip() { mb ^= 1; }
};

// Copy row elements [lo, lo + n) of `row` into shared memory at `dst`
// (16-byte aligned at element `head`), returning the largest packed
// (key, ~id) of the slice.  Vector loads where the global address allows.
template <typename T>
__device__ uint64_t load_slice(const T* __restrict__ row, int lo, int n, T* dst) {
  constexpr int kPer = 16 / sizeof(T);
  const T* g = row + lo;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(g) & 15u;
  int head = mis ? int((16u - mis) / sizeof(T)) : 0;
  if (head > n) head = n;
  const int nvec = (n - head) / kPer;
  const int tail0 = head + nvec * kPer;
  uint64_t best = 0;
  for (int i = threadIdx.x; i < head; i += kThreads) {
    const T v = g[i];
    dst[i] = v;
    const uint64_t p = pack_key_id(elem_key<T>(v), uint32_t(lo + i));
    best = p > best ? p : best;
  }
  const uint4* gv = reinterpret_cast<const uint4*>(g + head);
  uint4* sv = reinterpret_cast<uint4*>(dst + head);
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    const uint4 x = __ldg(gv + v);
    sv[v] = x;
    const T* e = reinterpret_cast<const T*>(&x);
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint64_t p = pack_key_id(elem_key<T>(e[j]), uint32_t(lo + head + v * kPer + j));
      best = p > best ? p : best;
    }
  }
  for (int i = tail0 + threadIdx.x; i < n; i += kThreads) {
    const T v = g[i];
    dst[i] = v;
    const uint64_t p = pack_key_id(elem_key<T>(v), uint32_t(lo + i));
    best = p > best ? p : best;
  }
  return best;
}

// Byte offset at which a slice starting at global element `row + lo` must be
// placed in shared memory so that its vector part is 16-byte aligned.
template <typename T>
__device__ __forceinline__ int slice_smem_offset(const T* row, int lo, int n) {
  const uintptr_t mis = reinterpret_cast<uintptr_t>(row + lo) & 15u;
  int head = mis ? int((16u - mis) / sizeof(T)) : 0;
  if (head > n) head = n;
  return int((16 - (head * int(sizeof(T))) % 16) % 16);
}

// Cluster-wide maximum of packed (key, ~id).
template <typename T>
__device__ uint64_t cluster_max(RowCtx<T>& c, uint64_t local) {
  local = block_max_u64(local, c.sh->red64);
  if (threadIdx.x == 0) c.mine().w[0] = local;
  c.exchange();
  uint64_t best = 0;
  if (c.alive) {
    for (uint32_t r = 0; r < c.nranks; ++r) {
      const uint64_t v = ld_cluster_u64(c.peer_addr(&c.mine().w[0], r));
      best = v > best ? v : best;
    }
  }
  c.flip();
  return best;
}

// Cluster-wide sums of up to 4 per-thread u64 values; also this CTA's own sum
// and the exclusive prefix over ranks of value 0.
template <typename T>
__device__ void cluster_sum4(RowCtx<T>& c, uint64_t v[4], int nv, uint64_t* prefix0,
                             uint64_t* local0 = nullptr) {
  for (int j = 0; j < nv; ++j) v[j] = block_sum<uint64_t>(v[j], c.sh->red64);
  if (local0) *local0 = v[0];
  if (threadIdx.x == 0)
    for (int j = 0; j < nv; ++j) c.mine().w[j] = v[j];
  c.exchange();
  uint64_t tot[4] = {0, 0, 0, 0};
  uint64_t pre = 0;
  if (c.alive) {
    for (uint32_t r = 0; r < c.nranks; ++r) {
      for (int j = 0; j < nv; ++j) {
        const uint64_t x = ld_cluster_u64(c.peer_addr(&c.mine().w[j], r));
        tot[j] += x;
        if (j == 0 && r < c.rank) pre += x;
      }
    }
  }
  for (int j = 0; j < nv; ++j) v[j] = tot[j];
  if (prefix0) *prefix0 = pre;
  c.flip();
}

// Cluster-wide sum of one u128 value and the exclusive prefix for this CTA.
template <typename T>
__device__ u128 cluster_sum128(RowCtx<T>& c, u128 local, u128* prefix) {
  local = block_sum<u128>(local, c.sh->red128);
  if (threadIdx.x == 0) c.mine().x[0] = local;
  c.exchange();
  u128 tot = 0, pre = 0;
  if (c.alive) {
    for (uint32_t r = 0; r < c.nranks; ++r) {
      const uint64_t lo = ld_cluster_u64(c.peer_addr(&c.mine().x[0], r));
      const uint64_t hi = ld_cluster_u64(c.peer_addr(reinterpret_cast<const char*>(&c.mine().x[0]) + 8, r));
      const u128 x = (u128(hi) << 64) | lo;
      tot += x;
      if (r < c.rank) pre += x;
    }
  }
  if (prefix) *prefix = pre;
  c.flip();
  return tot;
}

// Smallest global id over the cluster (0xFFFFFFFF if none).
template <typename T>
__device__ uint32_t cluster_min_id(RowCtx<T>& c, uint32_t local) {
  if (threadIdx.x == 0) c.mine().w[0] = local;
  c.exchange();
  uint32_t best = 0xFFFFFFFFu;
  if (c.alive) {
    for (uint32_t r = 0; r < c.nranks; ++r) {
      const uint32_t v = uint32_t(ld_cluster_u64(c.peer_addr(&c.mine().w[0], r)));
      best = v < best ? v : best;
    }
  }
  c.flip();
  return best;
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

// Result of selecting the boundary of a prefix of (key desc, id asc).
struct Boundary {
  uint32_t key;          // boundary key
  uint32_t n;            // members of the key's tie bucket in the prefix (>= 1)
  uint32_t above;        // elements with a larger key
  uint32_t tie_total;    // members of the tie bucket in the row
  uint32_t tie_base;     // tie members in lower-ranked CTAs
  uint32_t tie_local;    // tie members in this CTA
};

// Radix select over the slice keys, MSB-first 8-bit digits.
// kMass = false: the prefix of length `k`.
// kMass = true:  the shortest prefix whose mass reaches `target`.
template <typename T, bool kMass>
__device__ Boundary radix_select(RowCtx<T>& c, uint32_t k, const MassTarget& target,
                                 const RowScale& rs) {
  RowShared* sh = c.sh;
  const int tid = threadIdx.x;
  constexpr int kL = KeyTraits<T>::kLevels;
  uint32_t prefix = 0;
  uint32_t above = 0;
  uint64_t mass_above = 0;
  uint32_t my_rank_cnt[kMaxCluster];
  Boundary out;
  for (int lvl = 0; lvl < kL; ++lvl) {
    const int shift = 8 * (kL - 1 - lvl);
    sh->hist_cnt[tid] = 0;
    if (kMass) sh->hist_mass[tid] = 0;
    cta_sync();
    for (int i = tid; i < c.n; i += kThreads) {
      const uint32_t key = elem_key<T>(c.s[i]);
      if (lvl > 0 && (key >> (shift + 8)) != prefix) continue;
      const uint32_t d = (key >> shift) & 255u;
      atomicAdd(&sh->hist_cnt[d], 1u);
      if (kMass) {
        const uint64_t e = mass_fixed(Elem<T>::widen(c.s[i]), rs, c.table);
        if (e) atomicAdd(reinterpret_cast<unsigned long long*>(&sh->hist_mass[d]), (unsigned long long)e);
      }
    }
    cta_sync();
    c.mine().count[tid] = sh->hist_cnt[tid];
    if (kMass) c.mine().mass[tid] = sh->hist_mass[tid];
    c.exchange();
    uint32_t tc = 0;
    uint64_t tm = 0;
    if (c.alive) {
      for (uint32_t r = 0; r < c.nranks; ++r) {
        const uint32_t x = ld_cluster_u32(c.peer_addr(&c.mine().count[tid], r));
        my_rank_cnt[r] = x;
        tc += x;
        if (kMass) tm += ld_cluster_u64(c.peer_addr(&c.mine().mass[tid], r));
      }
    }
    sh->tot_cnt[tid] = tc;
    if (kMass) sh->tot_mass[tid] = tm;
    cta_sync();
    // Warp 0 finds the crossing digit, scanning digits from 255 down.
    if (tid < 32) {
      const int lane = tid;
      uint32_t lc = 0;
      uint64_t lm = 0;
      for (int j = 0; j < 8; ++j) {
        const int d = 255 - (lane * 8 + j);
        lc += sh->tot_cnt[d];
        if (kMass) lm += sh->tot_mass[d];
      }
      const uint32_t ic = warp_inclusive_scan<uint32_t>(lc);
      const uint64_t im = kMass ? warp_inclusive_scan<uint64_t>(lm) : 0;
      uint32_t run_c = above + ic - lc;
      uint64_t run_m = mass_above + im - lm;
      int found = -1;
      uint32_t found_above = 0;
      uint64_t found_mass_above = 0;
      for (int j = 0; j < 8 && found < 0; ++j) {
        const int d = 255 - (lane * 8 + j);
        const uint32_t nc = run_c + sh->tot_cnt[d];
        const uint64_t nm = kMass ? run_m + sh->tot_mass[d] : 0;
        bool hit;
        if (kMass) hit = sh->tot_cnt[d] > 0 && (target.trivial || mass_reaches(nm, target));
        else hit = nc >= k;
        if (hit) {
          found = d;
          found_above = run_c;
          found_mass_above = run_m;
        }
        run_c = nc;
        run_m = nm;
      }
      const uint32_t hits = __ballot_sync(0xFFFFFFFFu, found >= 0);
      // If nothing crossed (rounding cannot cause this with exact integers, but
      // guard anyway) take the last non-empty digit.
      int src = hits ? (__ffs(hits) - 1) : -1;
      if (src < 0) {
        int last = -1;
        for (int j = 0; j < 8; ++j) {
          const int d = 255 - (lane * 8 + j);
          if (sh->tot_cnt[d]) last = d;
        }
        const uint32_t nz = __ballot_sync(0xFFFFFFFFu, last >= 0);
        src = nz ? (31 - __clz(nz)) : 0;
        if (lane == src) {
          found = last < 0 ? 0 : last;
          uint32_t ca = 0;
          uint64_t ma = 0;
          for (int d = 255; d > found; --d) {
            ca += sh->tot_cnt[d];
            if (kMass) ma += sh->tot_mass[d];
          }
          found_above = above + ca;
          found_mass_above = mass_above + ma;
        }
      }
      if (lane == src) {
        sh->bcast32[0] = uint32_t(found);
        sh->bcast32[1] = found_above;
        sh->bcast64[0] = found_mass_above;
      }
    }
    cta_sync();
    const uint32_t d = sh->bcast32[0];
    above = sh->bcast32[1];
    mass_above = sh->bcast64[0];
    prefix = (prefix << 8) | d;
    if (lvl == kL - 1 && tid == int(d)) {
      for (uint32_t r = 0; r < c.nranks; ++r) sh->rank_cnt[r] = my_rank_cnt[r];
    }
    cta_sync();
    c.flip();
  }
  out.key = prefix;
  out.above = above;
  const uint32_t bucket = prefix & 255u;
  out.tie_total = sh->tot_cnt[bucket];
  out.tie_base = 0;
  for (uint32_t r = 0; r < c.rank; ++r) out.tie_base += sh->rank_cnt[r];
  out.tie_local = sh->rank_cnt[c.rank];
  if (!kMass) {
    out.n = k - above;
  } else {
    const uint64_t bucket_mass = sh->tot_mass[bucket];
    const uint64_t e_tie = out.tie_total ? bucket_mass / out.tie_total : 0;
    uint32_t n = 1;
    if (!target.trivial && e_tie > 0) {
      const u128 have = u128(mass_above) << target.sh;
      if (target.rhs > have) {
        // smallest n in [1, tie_total] with n * step >= need
        const u128 need = target.rhs - have;
        const u128 step = u128(e_tie) << target.sh;
        uint32_t lo_n = 1, hi_n = out.tie_total;
        while (lo_n < hi_n) {
          const uint32_t mid = lo_n + (hi_n - lo_n) / 2;
          if (u128(mid) * step >= need) hi_n = mid;
          else lo_n = mid + 1;
        }
        n = lo_n;
      }
    }
    out.n = n;
  }
  cta_sync();
  return out;
}

// The global id of the q-th (1-based) element with key == `key` in this CTA's
// slice, in id order; every thread gets the result.  Threads own contiguous
// chunks of the slice.
template <typename T>
__device__ uint32_t nth_with_key(RowCtx<T>& c, uint32_t key, uint32_t q) {
  RowShared* sh = c.sh;
  const int chunk = ((c.n + kThreads - 1) / kThreads) | 1;
  const int b0 = threadIdx.x * chunk;
  const int b1 = min(c.n, b0 + chunk);
  uint32_t cnt = 0;
  for (int i = b0; i < b1; ++i) cnt += elem_key<T>(c.s[i]) == key;
  // exclusive scan of counts over threads
  const uint32_t inc = warp_inclusive_scan<uint32_t>(cnt);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  cta_sync();
  if (lane == 31) sh->red32[warp] = inc;
  cta_sync();
  uint32_t before = inc - cnt;
  for (int w = 0; w < warp; ++w) before += sh->red32[w];
  if (threadIdx.x == 0) sh->bcast32[4] = 0xFFFFFFFFu;
  cta_sync();
  if (before < q && q <= before + cnt) {
    uint32_t seen = before;
    for (int i = b0; i < b1; ++i) {
      if (elem_key<T>(c.s[i]) == key && ++seen == q) {
        sh->bcast32[4] = uint32_t(c.lo + i);
        break;
      }
    }
  }
  cta_sync();
  return sh->bcast32[4];
}

// Weighted id-order search in this CTA's slice: the first element i for which
// the running sum of weight(i) exceeds `t` (t < total of the slice).  Threads
// own contiguous chunks; weight(i) is a functor of the slice index.
template <typename T, typename W, typename F>
__device__ int find_crossing(RowCtx<T>& c, W t, F weight, W* scratch_red, int* result) {
  const int chunk = ((c.n + kThreads - 1) / kThreads) | 1;
  const int b0 = threadIdx.x * chunk;
  const int b1 = min(c.n, b0 + chunk);
  W sum = 0;
  for (int i = b0; i < b1; ++i) sum += weight(i);
  const W inc = warp_inclusive_scan<W>(sum);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  cta_sync();
  if (lane == 31) scratch_red[warp] = inc;
  if (threadIdx.x == 0) *result = -1;
  cta_sync();
  W before = inc - sum;
  for (int w = 0; w < warp; ++w) before += scratch_red[w];
  if (sum > 0 && before <= t && t < before + sum) {
    W run = before;
    for (int i = b0; i < b1; ++i) {
      run += weight(i);
      if (run > t) {
        *result = i;
        break;
      }
    }
  }
  cta_sync();
  return *result;
}

}  // namespace smp
