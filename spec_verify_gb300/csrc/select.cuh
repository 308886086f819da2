// Exact selection of a row's kept set, shared by the sampler's general path
// and the verifier's filtered rows ("Decoding & Speculative Sampling",
// section 39.2 and eq. 39.2): knob rules, the min-p threshold key, passes over
// a row in global memory, MSB-first radix selection over order keys, the
// ranked candidate list for top-k up to kTopKMax, and the kept set S = the
// shortest of the enabled prefixes of the order (logit descending, id
// ascending) with its exact fixed-point mass Z_S.
//
// Every pass reads the row as 16-byte vectors.  A sweep (no order) keeps kU
// per thread in flight, vector base + u * kThreads + t for thread t, so each
// load instruction is coalesced.  A walk (id order) reads rounds of
// kThreads * kGenU vectors, thread t owning kGenU consecutive ones, so that
// (round, thread, vector, element) is token-id order.  Histograms are
// private per warp (count histograms for top-k, count and exact fixed-point
// mass histograms for top-p).
//
// Included inside namespace smp after row_ops.cuh.
#pragma once

// ------------------------------------------------------------------ knobs

__device__ __forceinline__ bool sampling_params_valid(const smp_row_params& p) {
  const float t = p.temperature;
  if (!(isfinite(t) && t > 0.0f)) return false;
  if (p.top_k < 0) return false;
  if (isnan(p.top_p) || p.top_p < 0.0f) return false;
  if (isnan(p.min_p) || p.min_p < 0.0f) return false;
  return true;
}

__device__ __forceinline__ bool row_is_greedy(const smp_row_params& p) {
  return p.greedy != 0 || p.temperature == 0.0f;
}

// ------------------------------------------------------------------ CTA helpers

// Sum of one u32 per thread over the CTA (every thread gets it).
__device__ __forceinline__ uint32_t block_sum_u32(uint32_t v, uint32_t* scratch) {
  v = warp_sum<uint32_t>(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  cta_sync();
  if (lane == 0) scratch[warp] = v;
  cta_sync();
  uint32_t t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += scratch[w];
  return t;
}

// Smallest key whose value z satisfies exp((z - m) / T) >= min_p, i.e. the
// min-p threshold p_i >= min_p * max_j p_j ("Inference: Sampling, the KV
// Cache, Speculative Decoding and int8", section "Picking the next token")
// expressed on logits.  Warp 0 probes 32 keys per step, starting around the
// estimate m + T ln(min_p); every thread gets the result.
template <typename T>
__device__ uint32_t minp_threshold_key(uint32_t* bcast, const FloatPair* table, const RowScale& rs, float temperature,
                                       float min_p, uint32_t key_max) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const double thr = double(min_p);
    const float est = rs.m + temperature * logf(min_p);
    const uint32_t k0 = KeyTraits<T>::kBits == 32 ? key_of_bits(__float_as_uint(est))
                                                  : (key_of_bits(__float_as_uint(est) & 0xFFFF0000u) >> 16);
    uint32_t lo = 0, hi = key_max;   // the answer lies in [lo, hi]; the property holds at hi
    uint32_t start = k0 > 16u ? k0 - 16u : 0u;
    uint32_t stride = 1;
    if (start > hi) start = hi;
    for (int iter = 0; iter < 64 && lo < hi; ++iter) {
      const uint64_t cand64 = uint64_t(start) + uint64_t(lane) * stride;
      const uint32_t cand = cand64 > hi ? hi : uint32_t(cand64);
      const bool ok = mass_double(key_value<T>(cand), rs, table) >= thr;
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, ok);
      const uint32_t last = __shfl_sync(0xFFFFFFFFu, cand, 31);
      if (mask == 0) {
        lo = last + 1 > hi ? hi : last + 1;
      } else {
        const int j = __ffs(mask) - 1;
        const uint32_t cj = __shfl_sync(0xFFFFFFFFu, cand, j);
        const uint32_t cprev = __shfl_sync(0xFFFFFFFFu, cand, j > 0 ? j - 1 : 0);
        hi = cj;
        if (j > 0) lo = cprev + 1;
        else if (start <= lo) lo = cj;   // probes started at the bottom of the range
      }
      if (lo > hi) lo = hi;
      const uint64_t span = uint64_t(hi - lo) + 1;
      stride = uint32_t((span + 31) / 32);
      start = lo;
    }
    if (lane == 0) bcast[6] = hi;
  }
  cta_sync();
  const uint32_t r = bcast[6];
  cta_sync();
  return r;
}

// ------------------------------------------------------------------ passes and radix selection

// 16-byte vectors per thread and round.  One keeps the exact exponential of
// every element inlined without spilling next to the candidate path's state.
constexpr int kGenU = 1;

// Shared state of the general path.
struct GenShared {
  uint32_t cnt[kWarps][256];
  // Fixed-point masses as three 15-bit limbs, each summed with 32-bit adds
  // (per warp and digit below 2^15 * 2^16 = 2^31 for V <= 2^19).
  uint32_t mass[kWarps][3][256];
  uint32_t tot_cnt[256];
  unsigned long long tot_mass[256];
  unsigned long long scan64[kWarps];
  uint32_t scan32[kWarps];
  uint64_t red64[kWarps];
  uint32_t bc32[8];
  unsigned long long bc64[4];
};

// Per-element transform of a row's logits, applied to every value a pass
// reads: xf(id, z) -> the logit the method sees.  NoPrep leaves it as is.
struct NoPrep {
  __device__ __forceinline__ float operator()(int, float z) const { return z; }
};

// Sweep over every element of a row in no particular order: f(id, xf(id, z)).
// kU vectors per thread in flight (more for light f).
template <typename T, int kU = kGenU, typename F, typename Xf = NoPrep>
__device__ __forceinline__ void gen_sweep(const T* row, int V, F&& f, const Xf& xf = Xf()) {
  using Vo = VecOps<T>;
  constexpr int kPer = Vo::kPer;
  const uintptr_t r0 = reinterpret_cast<uintptr_t>(row);
  const uintptr_t a0 = (r0 + 15) & ~uintptr_t(15), a1 = (r0 + size_t(V) * sizeof(T)) & ~uintptr_t(15);
  const bool mid = a1 > a0;
  const int head = mid ? int((a0 - r0) / sizeof(T)) : V;
  const int tail0 = mid ? int((a1 - r0) / sizeof(T)) : V;
  const int nvec = mid ? int((a1 - a0) / 16) : 0;
  const uint4* vp = reinterpret_cast<const uint4*>(a0);
  // vector base + u * kThreads + t for thread t: each load instruction coalesced
  for (int base = 0; base < nvec; base += kThreads * kU) {
    uint4 x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = base + u * kThreads + int(threadIdx.x);
      if (v < nvec) x[u] = __ldg(vp + v);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = base + u * kThreads + int(threadIdx.x);
      if (v < nvec) {
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
          const int id = head + v * kPer + q;
          f(id, xf(id, Vo::elem(x[u], q)));
        }
      }
    }
  }
  for (int i = threadIdx.x; i < head; i += kThreads) f(i, xf(i, Elem<T>::widen(row[i])));
  for (int i = tail0 + threadIdx.x; i < V; i += kThreads) f(i, xf(i, Elem<T>::widen(row[i])));
}

// Exclusive prefix over the CTA (thread order) of one value per thread, and the total.
template <typename U>
__device__ __forceinline__ U gen_scan(U v, U* warp_tot, U* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const U incl = warp_inclusive_scan<U>(v);
  if (lane == 31) warp_tot[warp] = incl;
  cta_sync();
  U before = incl - v, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const U t = warp_tot[w];
    if (w < warp) before += t;
    all += t;
  }
  cta_sync();
  *total = all;
  return before;
}

// Walk of a row in token-id order until the running value of g(id, z) passes
// `target` (strictly): returns that id, or -1.  g >= 0.  Each round is summed
// per thread, scanned over the CTA, and the thread whose interval holds the
// target walks its elements.  Elements before and after the aligned middle
// come first and last, walked by thread 0.
template <typename T, typename U, typename G, typename Xf = NoPrep>
__device__ int gen_walk(const T* row, int V, U target, GenShared& gs, G&& g, const Xf& xf = Xf()) {
  using Vo = VecOps<T>;
  constexpr int kPer = Vo::kPer;
  const uintptr_t r0 = reinterpret_cast<uintptr_t>(row);
  const uintptr_t a0 = (r0 + 15) & ~uintptr_t(15), a1 = (r0 + size_t(V) * sizeof(T)) & ~uintptr_t(15);
  const bool mid = a1 > a0;
  const int head = mid ? int((a0 - r0) / sizeof(T)) : V;
  const int tail0 = mid ? int((a1 - r0) / sizeof(T)) : V;
  const int nvec = mid ? int((a1 - a0) / 16) : 0;
  const uint4* vp = reinterpret_cast<const uint4*>(a0);
  U* warp_tot = reinterpret_cast<U*>(sizeof(U) == 8 ? static_cast<void*>(gs.scan64) : static_cast<void*>(gs.scan32));
  U run = 0;
  cta_sync();   // the previous reader of bc32[4] is done
  if (threadIdx.x == 0) gs.bc32[4] = 0xFFFFFFFFu;
  // head, by thread 0 (fewer than 16 / sizeof(T) elements, or the whole short row)
  if (threadIdx.x == 0) {
    U r = 0;
    for (int i = 0; i < head; ++i) {
      r += g(i, xf(i, Elem<T>::widen(row[i])));
      if (r > target) {
        gs.bc32[4] = uint32_t(i);
        break;
      }
    }
    gs.bc64[3] = (unsigned long long)r;
  }
  cta_sync();
  if (gs.bc32[4] != 0xFFFFFFFFu) return int(gs.bc32[4]);
  run = U(gs.bc64[3]);
  for (int base = 0; base < nvec; base += kThreads * kGenU) {
    const int v0 = base + threadIdx.x * kGenU;
    uint4 x[kGenU];
#pragma unroll
    for (int u = 0; u < kGenU; ++u)
      if (v0 + u < nvec) x[u] = __ldg(vp + v0 + u);
    U mine = 0;
#pragma unroll
    for (int u = 0; u < kGenU; ++u)
      if (v0 + u < nvec) {
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
          const int id = head + (v0 + u) * kPer + q;
          mine += g(id, xf(id, Vo::elem(x[u], q)));
        }
      }
    U total;
    const U before = run + gen_scan<U>(mine, warp_tot, &total);
    if (mine > 0 && before <= target && target - before < mine) {
      U r = before;
      bool done = false;
      for (int u = 0; u < kGenU && v0 + u < nvec && !done; ++u) {
        const uint4 xv = __ldg(vp + v0 + u);   // again, so that x stays in registers
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
          const int id = head + (v0 + u) * kPer + q;
          r += done ? U(0) : g(id, xf(id, Vo::elem(xv, q)));
          if (!done && r > target) {
            gs.bc32[4] = uint32_t(id);
            done = true;
          }
        }
      }
    }
    cta_sync();
    if (gs.bc32[4] != 0xFFFFFFFFu) return int(gs.bc32[4]);
    run += total;
  }
  if (threadIdx.x == 0) {
    U r = run;
    for (int i = tail0; i < V; ++i) {
      r += g(i, xf(i, Elem<T>::widen(row[i])));
      if (r > target) {
        gs.bc32[4] = uint32_t(i);
        break;
      }
    }
  }
  cta_sync();
  return gs.bc32[4] == 0xFFFFFFFFu ? -1 : int(gs.bc32[4]);
}

// Boundary of a prefix of (key desc, id asc): the boundary key, the elements
// above it, how many of its tie bucket are in the prefix, the bucket's size
// and, with masses, the fixed-point mass above the key.
struct GenBoundary {
  uint32_t key;
  uint32_t above;
  uint32_t n;
  uint32_t ties;
  uint64_t mass_above;
  uint64_t tie_mass;   // mass of one member of the tie bucket
};

// Radix selection, MSB-first 8-bit digits.  kMass = false: the prefix of
// length k (counts only).  kMass = true: the shortest prefix whose mass
// reaches the top-p target top_p * Z; the first level's mass total is Z,
// returned in *z_total.
template <typename T, bool kMass, typename Xf = NoPrep>
__device__ GenBoundary gen_select(const T* row, int V, GenShared& gs, uint32_t k, float top_p,
                                  const RowScale& rs, const FloatPair* table, uint64_t* z_total,
                                  const Xf& xf = Xf()) {
  constexpr int kL = KeyTraits<T>::kLevels;
  constexpr int kBits = KeyTraits<T>::kBits;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint32_t prefix = 0, above = 0;
  uint64_t mass_above = 0;
  MassTarget target{};
  for (int lvl = 0; lvl < kL; ++lvl) {
    const int shift = kBits - 8 * (lvl + 1);
    // Every bin of the last level is one key, whose elements share one mass:
    // that level counts, and a bin's mass is its count times the key's mass.
    const bool sweep_mass = kMass && lvl < kL - 1;
    for (int i = tid; i < kWarps * 256; i += kThreads) {
      (&gs.cnt[0][0])[i] = 0;
      if (sweep_mass) {
        (&gs.mass[0][0][0])[3 * i] = 0;
        (&gs.mass[0][0][0])[3 * i + 1] = 0;
        (&gs.mass[0][0][0])[3 * i + 2] = 0;
      }
    }
    cta_sync();
    gen_sweep<T>(row, V, [&](int, float z) {
      const uint32_t key = kBits == 32 ? key_of_bits(__float_as_uint(z)) : (key_of_bits(__float_as_uint(z)) >> 16);
      if (lvl > 0 && (key >> (shift + 8)) != prefix) return;
      const uint32_t d = (key >> shift) & 255u;
      atomicAdd(&gs.cnt[warp][d], 1u);
      if (sweep_mass) {
        const uint64_t e = mass_fixed(z, rs, table);
        if (e) {
          atomicAdd(&gs.mass[warp][0][d], uint32_t(e) & 0x7FFFu);
          atomicAdd(&gs.mass[warp][1][d], uint32_t(e >> 15) & 0x7FFFu);
          atomicAdd(&gs.mass[warp][2][d], uint32_t(e >> 30));
        }
      }
    }, xf);
    cta_sync();
    {   // one digit per thread: sum the warps' histograms
      uint32_t c = 0;
      unsigned long long mm = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        c += gs.cnt[w][tid];
        if (sweep_mass)
          mm += (unsigned long long)gs.mass[w][0][tid] + ((unsigned long long)gs.mass[w][1][tid] << 15) +
                ((unsigned long long)gs.mass[w][2][tid] << 30);
      }
      if (kMass && !sweep_mass && c)
        mm = (unsigned long long)c * mass_fixed(key_value<T>((prefix << 8) | uint32_t(tid)), rs, table);
      gs.tot_cnt[tid] = c;
      if (kMass) gs.tot_mass[tid] = mm;
    }
    cta_sync();
    if (kMass && lvl == 0) {
      // Z is the first level's total; the target compares exactly in 128 bits.
      if (tid < 32) {
        unsigned long long zz = 0;
        for (int j = 0; j < 8; ++j) zz += gs.tot_mass[lane * 8 + j];
        zz = warp_sum<uint64_t>(zz);
        if (lane == 0) gs.bc64[2] = zz;
      }
      cta_sync();
      *z_total = gs.bc64[2];
      target = make_mass_target(top_p, *z_total);
    }
    // Warp 0 finds the crossing digit, from 255 down.
    if (tid < 32) {
      uint32_t lc = 0;
      uint64_t lm = 0;
      for (int j = 0; j < 8; ++j) {
        const int d = 255 - (lane * 8 + j);
        lc += gs.tot_cnt[d];
        if (kMass) lm += gs.tot_mass[d];
      }
      const uint32_t ic = warp_inclusive_scan<uint32_t>(lc);
      const uint64_t im = kMass ? warp_inclusive_scan<uint64_t>(lm) : 0;
      uint32_t run_c = above + ic - lc;
      uint64_t run_m = mass_above + im - lm;
      int found = -1;
      uint32_t f_above = 0;
      uint64_t f_mass = 0;
      int last = -1;
      uint32_t l_above = 0;
      uint64_t l_mass = 0;
      for (int j = 0; j < 8; ++j) {
        const int d = 255 - (lane * 8 + j);
        const uint32_t c = gs.tot_cnt[d];
        const uint32_t nc = run_c + c;
        const uint64_t nm = kMass ? run_m + gs.tot_mass[d] : 0;
        if (c) {
          last = d;
          l_above = run_c;
          l_mass = run_m;
        }
        const bool hit = kMass ? (c > 0 && (target.trivial || mass_reaches(nm, target))) : (nc >= k);
        if (hit && found < 0) {
          found = d;
          f_above = run_c;
          f_mass = run_m;
        }
        run_c = nc;
        run_m = nm;
      }
      const uint32_t hits = __ballot_sync(0xFFFFFFFFu, found >= 0);
      int src;
      if (hits) {
        src = __ffs(hits) - 1;
      } else {
        // Nothing crossed (only possible through a degenerate target): the last non-empty digit.
        const uint32_t nz = __ballot_sync(0xFFFFFFFFu, last >= 0);
        src = nz ? 31 - __clz(nz) : 0;
        found = last < 0 ? 0 : last;
        f_above = l_above;
        f_mass = l_mass;
      }
      if (lane == src) {
        gs.bc32[0] = uint32_t(found);
        gs.bc32[1] = f_above;
        gs.bc64[0] = f_mass;
      }
    }
    cta_sync();
    const uint32_t d = gs.bc32[0];
    above = gs.bc32[1];
    mass_above = gs.bc64[0];
    prefix = (prefix << 8) | d;
    cta_sync();
  }
  GenBoundary out;
  out.key = prefix;
  out.above = above;
  out.ties = gs.tot_cnt[prefix & 255u];
  out.mass_above = mass_above;
  out.tie_mass = 0;
  if (!kMass) {
    out.n = k - above;
  } else {
    const uint64_t bucket_mass = gs.tot_mass[prefix & 255u];
    out.tie_mass = out.ties ? bucket_mass / out.ties : 0;   // every member has the same key, so the same mass
    uint32_t n = 1;
    if (!target.trivial && out.tie_mass > 0) {
      const u128 have = u128(mass_above) << target.sh;
      if (target.rhs > have) {
        // smallest n >= 1 with (mass_above + n * tie_mass) << sh >= rhs
        const u128 need = target.rhs - have;
        const u128 step = u128(out.tie_mass) << target.sh;
        uint32_t lo = 1, hi = out.ties;
        while (lo < hi) {
          const uint32_t mid = lo + (hi - lo) / 2;
          if (u128(mid) * step >= need) hi = mid;
          else lo = mid + 1;
        }
        n = lo;
      }
    }
    out.n = n > out.ties ? out.ties : n;
  }
  return out;
}

// ------------------------------------------------------------------ k-th largest of a short list

// The k-th largest (1 <= k <= n) of n keys key_at(0 .. n-1), exactly: radix
// selection over their top 8 * kLevels bits with 8-bit digits, one shared
// 256-bin histogram per level.  Returns those bits, right-aligned.
template <int kLevels, typename KeyAt>
__device__ uint32_t kth_largest_key(int n, uint32_t k, KeyAt&& key_at, uint32_t* hist, uint32_t* bcast) {
  uint32_t prefix = 0;
  uint32_t need = k;
  for (int lvl = 0; lvl < kLevels; ++lvl) {
    const int shift = 24 - 8 * lvl;
    hist[threadIdx.x] = 0;
    cta_sync();
    for (int i = threadIdx.x; i < n; i += kThreads) {
      const uint32_t key = key_at(i);
      if (lvl == 0 || (key >> (shift + 8)) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    cta_sync();
    if (threadIdx.x < 32) {
      // digits 255..0 in lane order: lane l covers 255 - 8l .. 248 - 8l
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - (threadIdx.x * 8 + j)];
        sum += c[j];
      }
      const uint32_t incl = warp_inclusive_scan<uint32_t>(sum);
      uint32_t run = incl - sum;
      int found = -1;
      uint32_t above = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (found < 0 && run + c[j] >= need) {
          found = 255 - (threadIdx.x * 8 + j);
          above = run;
        }
        run += c[j];
      }
      const uint32_t hits = __ballot_sync(0xFFFFFFFFu, found >= 0);
      const int src = hits ? __ffs(hits) - 1 : 0;
      if (threadIdx.x == src) {
        bcast[0] = uint32_t(found < 0 ? 0 : found);
        bcast[1] = above;
      }
    }
    cta_sync();
    prefix = (prefix << 8) | bcast[0];
    need -= bcast[1];
    cta_sync();
  }
  return prefix;
}

// The k-th largest of vals[0..n) (1 <= k <= n), exactly, as a float (two
// levels for bf16 values, four for binary32).
template <typename T>
__device__ float kth_largest_list(const float* vals, int n, int k, uint32_t* hist, uint32_t* bcast) {
  constexpr int kLevels = KeyTraits<T>::kBits == 16 ? 2 : 4;
  const uint32_t prefix = kth_largest_key<kLevels>(
      n, uint32_t(k), [&](int i) { return key_of_bits(__float_as_uint(vals[i])); }, hist, bcast);
  return value_of_key(kLevels == 2 ? (prefix << 16) | ((prefix & 0x8000u) ? 0u : 0xFFFFu) : prefix);
}

// ------------------------------------------------------------------ the kept set

// The kept set S of one row: token i with order key k_i is in S when
//   k_i > key, or k_i == key and i <= id_cut
// (every filter off: key 0, id_cut 0xFFFFFFFF, so every token is kept).
// Each enabled mask (top-k, top-p, min-p) is a prefix of the order (logit
// descending, id ascending), so their intersection is the shortest of them.
struct KeptSet {
  RowScale rs;       // row maximum and 1/T
  uint32_t key;
  uint32_t id_cut;
  uint64_t len;      // |S|
  uint64_t z_kept;   // Z_S: the sum of the kept tokens' fixed-point masses
};

template <typename T>
__device__ __forceinline__ uint32_t order_key(float z) {
  return KeyTraits<T>::kBits == 32 ? key_of_bits(__float_as_uint(z)) : (key_of_bits(__float_as_uint(z)) >> 16);
}

__device__ __forceinline__ bool in_kept_set(const KeptSet& ks, uint32_t key, uint32_t id) {
  return key > ks.key || (key == ks.key && id <= ks.id_cut);
}

// The fixed-point mass of token i (logit z) if it is kept, else 0.
template <typename T>
__device__ __forceinline__ uint64_t kept_mass(const KeptSet& ks, const FloatPair* table, int i, float z) {
  return in_kept_set(ks, order_key<T>(z), uint32_t(i)) ? mass_fixed(z, ks.rs, table) : 0ull;
}

// S and Z_S of a row whose maximum key is finite and whose knobs are valid
// sampling knobs (not greedy): the min-p threshold key, the radix selections
// of top-k and top-p, the tie member at the boundary (an id-order walk) and
// Z_S (from the top-p histograms when top-p set the boundary, else a pass).
// Every thread gets the result.
template <typename T, typename Xf = NoPrep>
__device__ KeptSet gen_kept_set(const T* row, int V, GenShared& gs, const FloatPair* table,
                                const smp_row_params& prm, uint32_t key_max, const Xf& xf = Xf()) {
  const int tid = threadIdx.x;
  KeptSet ks;
  ks.rs = make_row_scale(key_value<T>(key_max), prm.temperature);
  const bool topk = prm.top_k > 0 && prm.top_k < V;
  const bool topp = prm.top_p < 1.0f;
  const bool minp = prm.min_p > 0.0f && prm.min_p < 1.0f;

  // Prefix lengths of the enabled filters.
  uint64_t len_k = uint64_t(V), len_p = uint64_t(V), len_m = uint64_t(V);
  uint32_t key_min_p = 0;
  if (minp) {
    key_min_p = minp_threshold_key<T>(gs.bc32, table, ks.rs, prm.temperature, prm.min_p, key_max);
    uint32_t c = 0;
    gen_sweep<T>(row, V, [&](int, float z) { c += order_key<T>(z) >= key_min_p; }, xf);
    len_m = block_sum_u32(c, gs.scan32);
  }
  GenBoundary bk{}, bp{};
  uint64_t z_total = 0;
  if (topk) {
    bk = gen_select<T, false>(row, V, gs, uint32_t(prm.top_k), 1.0f, ks.rs, table, &z_total, xf);
    len_k = uint64_t(prm.top_k);
  }
  if (topp) {
    bp = gen_select<T, true>(row, V, gs, 0, prm.top_p, ks.rs, table, &z_total, xf);
    len_p = uint64_t(bp.above) + bp.n;
  }
  uint64_t len = len_k < len_p ? len_k : len_p;
  len = len < len_m ? len : len_m;
  ks.len = len;
  ks.key = 0;
  ks.id_cut = 0xFFFFFFFFu;
  GenBoundary bd{};
  bool from_p = false, cut = false;
  if (len < uint64_t(V)) {
    cut = true;
    if (minp && len == len_m) {
      ks.key = key_min_p;   // every token at or above the threshold key
    } else {
      from_p = !(topk && len == len_k);
      bd = from_p ? bp : bk;
      ks.key = bd.key;
      if (bd.n < bd.ties) {   // the id of the n-th member (id order) of the boundary's tie bucket
        const int id = gen_walk<T, uint32_t>(row, V, bd.n - 1, gs, [&](int, float z) -> uint32_t {
          return order_key<T>(z) == bd.key ? 1u : 0u;
        }, xf);
        ks.id_cut = uint32_t(id);
      }
    }
  }
  if (cut && from_p) {
    ks.z_kept = bd.mass_above + uint64_t(bd.n) * bd.tie_mass;
  } else if (!cut && topp) {
    ks.z_kept = z_total;
  } else {
    uint64_t zl = 0;
    gen_sweep<T>(row, V, [&](int i, float z) { zl += kept_mass<T>(ks, table, i, z); }, xf);
    zl = warp_sum<uint64_t>(zl);
    if ((tid & 31) == 0) gs.scan64[tid >> 5] = zl;
    cta_sync();
    uint64_t zk = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) zk += gs.scan64[w];
    cta_sync();
    ks.z_kept = zk;
  }
  return ks;
}

// ------------------------------------------------------------------ top-k-bounded kept set

// With top-k set to k <= kTopKMax the kept set holds at most k tokens, so it
// comes from a short candidate list instead of radix passes over the row.
// theta, the k-th largest of the threads' maximum keys from the caller's
// maximum pass (to 16 bits), bounds the row's k-th largest key from below
// (k threads each saw a key >= theta); one pass collects every token with key >= theta, and
// the candidates are ranked exactly by (key desc, id asc).  The first k get
// their exact fixed-point masses and prefix sums; min-p cuts at the first
// whose exponential falls below min_p; top-p compares the prefix sums with
// top_p * Z, Z bracketed by a binary32 sum of every token's exponential
// taken in the same pass (topk_z_bracket).  A prefix that falls inside the
// bracket asks for the exact Z, one more pass.  More than kTopCandMax candidates
// (long runs of equal keys) and the row takes gen_kept_set.
constexpr int kTopKMax = 128;
constexpr int kTopCandMax = 1024;
constexpr int kTopU = 4;   // vectors in flight per thread in the light passes (default)

// kU for raw rows; one vector in flight under a logit transform, whose
// state already fills the registers.
template <typename Xf, int kU = kTopU>
constexpr int light_pass_vectors() {
  return std::is_same<Xf, NoPrep>::value ? kU : 1;
}

static_assert(sizeof(GenShared::mass) >= sizeof(unsigned long long) * (kTopCandMax + 2 * kTopKMax),
              "candidate list, ranked list and masses overlay the mass histograms");

__device__ __forceinline__ unsigned long long* topk_cand(GenShared& gs) {
  return reinterpret_cast<unsigned long long*>(&gs.mass[0][0][0]);
}
// the first k candidates by rank, packed (key << 32) | ~id
__device__ __forceinline__ unsigned long long* topk_list(GenShared& gs) { return topk_cand(gs) + kTopCandMax; }
// their fixed-point masses
__device__ __forceinline__ unsigned long long* topk_mass(GenShared& gs) {
  return topk_cand(gs) + kTopCandMax + kTopKMax;
}

__device__ __forceinline__ bool topk_bounded(const smp_row_params& prm, int V) {
  return prm.top_k > 0 && prm.top_k <= kTopKMax && prm.top_k < V;
}

// The candidate pass of gen_kept_set_topk (also the beam step's slices, which
// ask for no sums).  Every token whose key is at
// least theta is appended to cand (a count past kTopCandMax is an overflow):
// raw rows compare the logit with theta's value (theta finite), transformed
// rows compare keys.  With top-p, each thread also sums e' = 2^y',
// y' = fl(fl(z - m) * c_hi), pairwise within each 16-byte vector and then one
// add per vector, and A = sum e' |y'|.  The bracket on Z follows from them
// (topk_z_bracket).
struct ZSums {
  float z;    // sum of e'
  float a;    // -(sum of e' |y'|)
};

template <typename T, int kU, bool kRaw, bool kTopp, typename Xf>
__device__ __forceinline__ ZSums topk_candidate_pass(const T* row, int V, uint32_t theta, float theta_v,
                                                     const RowScale& rs, unsigned long long* cand, uint32_t* count,
                                                     const Xf& xf) {
  using Vo = VecOps<T>;
  constexpr int kPer = Vo::kPer;
  const uintptr_t r0 = reinterpret_cast<uintptr_t>(row);
  const uintptr_t a0 = (r0 + 15) & ~uintptr_t(15), a1 = (r0 + size_t(V) * sizeof(T)) & ~uintptr_t(15);
  const bool mid = a1 > a0;
  const int head = mid ? int((a0 - r0) / sizeof(T)) : V;
  const int tail0 = mid ? int((a1 - r0) / sizeof(T)) : V;
  const int nvec = mid ? int((a1 - a0) / 16) : 0;
  const uint4* vp = reinterpret_cast<const uint4*>(a0);
  ZSums acc{0.0f, 0.0f};
  auto is_cand = [&](float z) -> bool { return kRaw ? (z >= theta_v) : (order_key<T>(z) >= theta); };
  auto append = [&](int id, float z) {
    const uint32_t s = atomicAdd(count, 1u);
    if (s < uint32_t(kTopCandMax)) cand[s] = pack_key_id(order_key<T>(z), uint32_t(id));
  };
  // e' of one logit (0 unless live); y clamped at -127 (also -inf and NaN),
  // where the flushed result is 0; acc.a gathers -sum e' |y'| (y <= 0)
  auto expo = [&](float z, bool live) -> float {
    const float y = fmaxf(__fmul_rn(__fsub_rn(z, rs.m), rs.c_hi), -127.0f);
    const float e = live ? ex2_approx(y) : 0.0f;
    acc.a = __fmaf_rn(e, y, acc.a);
    return e;
  };
  for (int base = 0; base < nvec; base += kThreads * kU) {
    uint4 x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = base + u * kThreads + int(threadIdx.x);
      x[u] = v < nvec ? __ldg(vp + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    // Every exponential first, free of branches, with a bit per candidate;
    // the candidates (rare) after, their logits read again one by one.
    static_assert(kU * kPer <= 64, "one bit per element of a round");
    unsigned long long bits = 0;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int v = base + u * kThreads + int(threadIdx.x);
      float ev[kPer];
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const float z = xf(head + v * kPer + q, Vo::elem(x[u], q));
        if (v < nvec && is_cand(z)) bits |= 1ull << (u * kPer + q);
        if (kTopp) ev[q] = expo(z, v < nvec);
      }
      if (kTopp) {
#pragma unroll
        for (int w = 1; w < kPer; w <<= 1)
#pragma unroll
          for (int q = 0; q + w < kPer; q += 2 * w) ev[q] = __fadd_rn(ev[q], ev[q + w]);
        acc.z = __fadd_rn(acc.z, ev[0]);
      }
    }
    if (__any_sync(0xFFFFFFFFu, bits != 0)) {
      // One atomic per warp: each lane's count, an exclusive scan over the
      // lanes, lane 31 reserves the warp's slots.
      const uint32_t mine = uint32_t(__popcll(bits));
      const uint32_t incl = warp_inclusive_scan<uint32_t>(mine);
      uint32_t slot = 0;
      if ((threadIdx.x & 31) == 31) slot = atomicAdd(count, incl);
      slot = __shfl_sync(0xFFFFFFFFu, slot, 31) + incl - mine;
      while (bits) {
        const int j = __ffsll((long long)bits) - 1;
        bits &= bits - 1;
        const int id = head + (base + (j / kPer) * kThreads + int(threadIdx.x)) * kPer + j % kPer;
        const float z = xf(id, Elem<T>::widen(row[id]));
        if (slot < uint32_t(kTopCandMax)) cand[slot] = pack_key_id(order_key<T>(z), uint32_t(id));
        ++slot;
      }
    }
  }
  auto one = [&](int i) {
    const float z = xf(i, Elem<T>::widen(row[i]));
    if (is_cand(z)) append(i, z);
    if (kTopp) acc.z = __fadd_rn(acc.z, expo(z, true));
  };
  for (int i = threadIdx.x; i < head; i += kThreads) one(i);
  for (int i = tail0 + threadIdx.x; i < V; i += kThreads) one(i);
  return acc;
}

// The bracket [z_lo, z_hi] on the exact fixed-point Z from the threads'
// ZSums (every thread gets it).  Errors, relative to each e = 2^y:
//  * y' against y: fl(z - m), log2(e) rounded to binary32, its quotient by
//    T rounded to c_hi, and the product: 4 units of 2^-24 of |y| in all, so
//    e' is off by at most ln 2 * 4.01 * 2^-24 |y| e, bounded through A
//    (2.8 * 2^-24 A);
//  * ex2.approx: taken within 2^-21 relative (its largest relative error over
//    every binary32 argument in [-126, 1], measured on GB300, is 1.46e-7);
//  * the sums: a thread adds at most log2(elements per vector) + its vectors
//    + 2 terms in sequence, a warp's lanes meet in a tree of depth 5 and
//    thread 0 adds the warps' sums in sequence, each add within 2^-24 of its
//    running sum;
//  * the fixed-point masses: 3/4 of a unit per token (rounding, and values
//    below 2^-47 dropped); tokens below 2^-126, dropped here, weigh less.
// Margins of 2^-9 cover the second-order terms; the bound itself is
// evaluated with upward rounding.
template <typename T>
__device__ __forceinline__ void topk_z_bracket(ZSums acc, int V, GenShared& gs, uint64_t* z_lo, uint64_t* z_hi) {
  constexpr int kLogPer = VecOps<T>::kPer == 8 ? 3 : VecOps<T>::kPer == 4 ? 2 : 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float zt = acc.z, at = -acc.a;
#pragma unroll
  for (int o = 16; o; o >>= 1) {   // a tree of depth 5 over the lanes
    zt = __fadd_rn(zt, __shfl_xor_sync(0xFFFFFFFFu, zt, o));
    at = __fadd_rn(at, __shfl_xor_sync(0xFFFFFFFFu, at, o));
  }
  float2* part = reinterpret_cast<float2*>(gs.scan64);
  if (lane == 0) part[warp] = make_float2(zt, at);
  cta_sync();
  if (threadIdx.x == 0) {
    // binary32 throughout (thread 0 alone), every rounding inside the margins
    float zf = 0.0f, af = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      zf = __fadd_rn(zf, part[w].x);
      af = __fadd_rn(af, part[w].y);
    }
    const int nvec = V * int(sizeof(T)) / 16 + 1;
    const float adds = float(kLogPer + (nvec + kThreads - 1) / kThreads + 2 + 5 + kWarps);
    const float u = 0x1p-24f;
    const float zd = __fmul_rn(zf, float(kFixedOne));   // exact
    const float rel = __fmul_ru(__fmaf_ru(adds, u, 0x1p-21f), 1.0f + 0x1p-9f);
    const float w = __fmul_ru(__fadd_ru(__fadd_ru(__fmul_ru(rel, zd),
                                                  __fmul_ru(__fmul_ru(2.8f * u, af), float(kFixedOne))),
                                        __fmaf_ru(0.75f, float(V), 2.0f)),
                              1.0f + 0x1p-9f);
    const float lo = __fsub_rd(zd, w);
    gs.bc64[1] = lo > 0.0f ? __float2ull_rd(lo) : 0ull;
    gs.bc64[2] = __float2ull_ru(__fadd_ru(zd, w));
  }
  cta_sync();
  *z_lo = gs.bc64[1];
  *z_hi = gs.bc64[2];
}

// S and Z_S of a row as gen_kept_set gives them, for a row with
// topk_bounded(prm, V), valid sampling knobs (not greedy) and a finite
// maximum key.  thread_key_max is this thread's maximum key in a pass over
// every element (any split of the row over the threads); kU is the number
// of vectors each thread keeps in flight in the candidate pass.  Returns
// false, with every thread agreeing, when the candidates overflow or fewer
// than k threads saw a finite maximum (raw rows).  On success the first
// ks.len entries of topk_list and topk_mass hold S in rank order.
template <typename T, int kU = kTopU, typename Xf = NoPrep>
__device__ bool gen_kept_set_topk(const T* row, int V, GenShared& gs, const FloatPair* table,
                                  const smp_row_params& prm, uint32_t key_max, uint32_t thread_key_max,
                                  KeptSet* out, const Xf& xf = Xf()) {
  constexpr int kKeyUp = 32 - KeyTraits<T>::kBits;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t k = uint32_t(prm.top_k);
  const bool topp = prm.top_p < 1.0f;
  const bool minp = prm.min_p > 0.0f && prm.min_p < 1.0f;
  KeptSet ks;
  ks.rs = make_row_scale(key_value<T>(key_max), prm.temperature);

  // theta: the top 16 bits of the k-th largest of the threads' maximum keys
  // (k <= kThreads), the rest zero: exact for bf16 keys, a lower bound one
  // bf16 step wide for binary32 keys, which only adds a few candidates.
  uint32_t* tkeys = &gs.cnt[0][0];
  cta_sync();   // earlier readers of the overlaid state are done
  tkeys[tid] = thread_key_max;
  const uint32_t theta = kth_largest_key<2>(kThreads, k, [&](int i) { return tkeys[i] << kKeyUp; },
                                             gs.tot_cnt, gs.bc32) << (16 - kKeyUp);

  // One pass: the candidates, and the sums of the bracket on Z.
  constexpr bool kRaw = std::is_same<Xf, NoPrep>::value;
  if (kRaw && !key_finite<T>(theta)) return false;   // fewer than k finite thread maxima
  unsigned long long* cand = topk_cand(gs);
  if (tid == 0) gs.bc32[5] = 0;
  cta_sync();
  constexpr int kPassU = light_pass_vectors<Xf, kU>();
  const ZSums acc =
      topp ? topk_candidate_pass<T, kPassU, kRaw, true>(row, V, theta, key_value<T>(theta), ks.rs, cand, &gs.bc32[5], xf)
           : topk_candidate_pass<T, kPassU, kRaw, false>(row, V, theta, key_value<T>(theta), ks.rs, cand, &gs.bc32[5], xf);
  cta_sync();
  const uint32_t n = gs.bc32[5];
  if (n > uint32_t(kTopCandMax) || n < k) {   // (n >= k whenever thread_key_max is as stated)
    cta_sync();
    return false;
  }
  uint64_t z_lo = 0, z_hi = 0;
  if (topp) topk_z_bracket<T>(acc, V, gs, &z_lo, &z_hi);

  // Rank every candidate; the first k by rank, in rank order.
  unsigned long long* list = topk_list(gs);
  unsigned long long* lmass = topk_mass(gs);
  for (int c = tid; c < int(n); c += kThreads) {
    const unsigned long long pc = cand[c];
    uint32_t r = 0;
    for (int j = 0; j < int(n); ++j) r += cand[j] > pc;
    if (r < k) list[r] = pc;
  }
  if (tid == 0) {
    gs.bc32[2] = k - 1;   // first rank whose prefix may reach the top-p target
    gs.bc32[3] = k - 1;   // first rank whose prefix surely reaches it
  }
  cta_sync();
  // Exact masses of the first k (their logits read again), and the min-p
  // test exp((z - m) / T) >= min_p on each (parts_at_least, exact).
  uint64_t e = 0;
  bool below_min_p = false;
  if (uint32_t(tid) < k) {
    const uint32_t id = ~uint32_t(list[tid]);
    const ExpParts ep = exp_parts(xf(int(id), Elem<T>::widen(row[id])), ks.rs, table, -1000.0f);
    e = fixed_from_parts(ep);
    lmass[tid] = e;
    below_min_p = minp && !parts_at_least(ep, prm.min_p);
  }
  // Masses fall along the ranks, so the tokens that pass min-p are the ranks
  // below the first that does not (the maximum always passes).
  const uint32_t len_m = k - uint32_t(cta_sync_count(below_min_p));
  uint64_t total;
  const uint64_t cum =   // prefix mass through this rank
      gen_scan<uint64_t>(e, reinterpret_cast<uint64_t*>(gs.scan64), &total) + e;

  // Top-p: the first rank r whose prefix reaches top_p * Z (only r < k - 1 matters).
  uint32_t len_p = k;
  if (topp) {
    const MassTarget t_lo = make_mass_target(prm.top_p, z_lo);   // reached first
    const MassTarget t_hi = make_mass_target(prm.top_p, z_hi);
    if (t_lo.trivial) {
      len_p = 1;
    } else {
      if (uint32_t(tid) + 1 < k) {
        if (mass_reaches(cum, t_lo)) atomicMin(&gs.bc32[2], uint32_t(tid));
        if (mass_reaches(cum, t_hi)) atomicMin(&gs.bc32[3], uint32_t(tid));
      }
      cta_sync();
      uint32_t first = gs.bc32[2];
      if (first != gs.bc32[3]) {
        // The bracket does not decide: the exact Z.
        uint64_t zz = 0;
        gen_sweep<T>(row, V, [&](int, float z) { zz += mass_fixed(z, ks.rs, table); }, xf);
        zz = warp_sum<uint64_t>(zz);
        cta_sync();
        if (lane == 0) gs.scan64[warp] = zz;
        if (tid == 0) gs.bc32[2] = k - 1;
        cta_sync();
        uint64_t z_exact = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) z_exact += gs.scan64[w];
        const MassTarget tx = make_mass_target(prm.top_p, z_exact);
        if (uint32_t(tid) + 1 < k && mass_reaches(cum, tx)) atomicMin(&gs.bc32[2], uint32_t(tid));
        cta_sync();
        first = gs.bc32[2];
      }
      len_p = first + 1;
    }
  }
  uint32_t len = k < len_p ? k : len_p;
  len = len < len_m ? len : len_m;
  if (uint32_t(tid) == len - 1) gs.bc64[0] = cum;
  cta_sync();
  const unsigned long long last = list[len - 1];
  ks.len = len;
  ks.key = uint32_t(last >> 32);
  ks.id_cut = ~uint32_t(last);
  ks.z_kept = gs.bc64[0];
  cta_sync();
  *out = ks;
  return true;
}
