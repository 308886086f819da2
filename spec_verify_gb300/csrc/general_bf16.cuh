// General path of the sampler for bf16 logits: any knobs (top-p, unfiltered
// sampling, any k), exactly, with one double-float exponential per distinct
// logit value instead of one per element ("Decoding & Speculative Sampling",
// section 39.2 and eq. 39.2; "Choosing the next word", section "Where the
// randomness comes from, and where it stops").
//
// A bf16 logit has one of 2^16 values, and tokens with the same value have
// the same mass.  So:
//
//   pass 1   (the row, from HBM)  the row maximum and, for every logit value
//            in a window of order keys that holds every value of nonzero mass,
//            the number of tokens with that value: one counter per key in
//            shared memory.  Values of very small magnitude (|z| below the
//            window's cutoff, zeros included) would need a counter for every
//            one of their many binades; the few tokens that hold them go to a
//            short list instead.  The window is anchored at an early estimate
//            of the maximum with room above it;
//   table    E(key) = round(exp((z - max z) / T) 2^44) by the double-float
//            exponential for every key that occurs; Z = sum count * E, exact;
//   select   top-k, top-p and min-p on the table in key order: scans of
//            counts and masses, the crossing found exactly in 128 bits, the
//            number n of tokens of the boundary key that are kept;
//   pass 2   (the row again, normally from L2)  the draw: token ids in order,
//            each token's mass looked up in the table, the boundary key's
//            first n tokens (id order) kept, rounds scanned over the CTA, the
//            crossing thread walking its ids.
//
// A row the table cannot take (a value above the window, more small-magnitude
// tokens than the list holds, or a boundary among them) returns false before
// it writes anything, and the caller runs the per-element path instead.
// Included by sample.cu inside namespace smp after general.cuh.
#pragma once

constexpr int kKtSlots = 4864;     // one counter per order key of the window's dense part
constexpr int kKtSparse = 256;     // tokens of small magnitude, listed one by one
constexpr int kKtU = 8;            // 16-byte vectors per thread and round

// Slots kKtSlots .. kKtSlots + 31 are per-lane dummies: a token outside the
// dense part is counted there (no branch per token) and has mass 0.
constexpr int kKtAll = kKtSlots + 32;

struct KeyTable {
  uint32_t cnt[kKtAll];
  unsigned long long mass[kKtAll];             // E of the slot's key, once the counts are in
  unsigned long long sparse[kKtSparse];        // (key << 32) | id of a small-magnitude token
  unsigned long long sparse_mass[kKtSparse];   // its E
  unsigned long long scan64[kWarps];
  uint32_t scan32[kWarps];
  uint64_t red64[kWarps];
  float redf[kWarps];
  uint32_t bc32[8];
  unsigned long long bc64[4];
  uint32_t sp_n;      // small-magnitude tokens seen
  int overflow;       // a token above the window, or too many small ones
  // the window: dense keys kposlo..kt (slots 0..nP-1, descending) and
  // kb..knhi (slots nP..nP+nN-1, descending); keys between knhi and kposlo
  // are the small magnitudes
  uint32_t kt, kposlo, knhi, kb;
  int nP, nN;
};
static_assert(sizeof(KeyTable) <= size_t(kBufs) * kBufBytes, "the key table overlays the idle ring");

__device__ __forceinline__ uint32_t key16_of(float z) { return key_of_bits(__float_as_uint(z)) >> 16; }

// u64 -> float within two roundings, from 32-bit conversions (the 64-bit
// conversion instructions run on the binary64 pipe, which is narrow on this
// part).
__device__ __forceinline__ float kt_u64_to_f(uint64_t x) {
  return __fmaf_rn(__uint2float_rn(uint32_t(x >> 32)), 0x1p32f, __uint2float_rn(uint32_t(x)));
}

// The window for an estimate m0 of the row maximum: keys above the key of
// m0 + 8 T would be tokens above the window (checked once the maximum is
// known); tokens with keys below the key of m0 - 33 T have
// exp((z - max) / T) < 2^-47 for any maximum >= m0, zero in 2^-44 units.  The
// cutoff of small magnitudes, 2^c, is the smallest that leaves the dense part
// within kKtSlots keys.  Thread 0; false if no cutoff fits.
__device__ __forceinline__ bool kt_window(KeyTable& kt, float m0, float temperature) {
  const float top = fminf(__fmaf_rn(8.0f, temperature, m0), 3.0e38f);
  const float bottom = fmaxf(__fmaf_rn(-33.0f, temperature, m0), -3.0e38f);
  const uint32_t ktop = min(key16_of(top) + 1u, 0xFF7Fu);
  const uint32_t kbot = max(key16_of(bottom), 0x0081u) - 1u;
  for (int c = -24; c <= 120; ++c) {
    const uint32_t e = uint32_t(127 + c) << 7;
    const uint32_t kposmin = 0x8000u | e;            // key of +2^c
    const uint32_t knegmax = ~(0x8000u | e) & 0xFFFFu;   // key of -2^c
    const uint32_t kposlo = max(kbot, kposmin);
    const int nP = ktop >= kposlo ? int(ktop - kposlo + 1) : 0;
    const uint32_t knhi = min(ktop, knegmax);
    const int nN = knhi >= kbot ? int(knhi - kbot + 1) : 0;
    if (nP + nN <= kKtSlots) {
      kt.kt = ktop;
      kt.kposlo = kposlo;
      kt.knhi = knhi;
      kt.kb = kbot;
      kt.nP = nP;
      kt.nN = nN;
      return true;
    }
  }
  return false;
}

// Dense slot of a key inside the window, or -1.
__device__ __forceinline__ int kt_slot(const KeyTable& kt, uint32_t key) {
  if (key >= kt.kposlo && key <= kt.kt) return int(kt.kt - key);
  if (key <= kt.knhi && key >= kt.kb) return kt.nP + int(kt.knhi - key);
  return -1;
}

// The order key of a bf16 bit pattern (-0 as +0, NaN as -inf).
__device__ __forceinline__ uint32_t kt_key_bits(uint32_t h) {
  h = h == 0x8000u ? 0u : h;
  const uint32_t k = (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
  return (h & 0x7FFFu) > 0x7F80u ? 0x007Fu : k;
}

// The slot of a key without branches: dense slot, or the lane's dummy.
__device__ __forceinline__ uint32_t kt_slot_nb(uint32_t kt_top, uint32_t knhi, uint32_t nP, uint32_t nN,
                                               uint32_t key, uint32_t lane) {
  const uint32_t dp = kt_top - key, dn = knhi - key;   // unsigned: out of range wraps to large
  return dp < nP ? dp : (dn < nN ? nP + dn : uint32_t(kKtSlots) + lane);
}

__device__ __forceinline__ uint32_t kt_key_of_slot(const KeyTable& kt, int s) {
  return s < kt.nP ? kt.kt - uint32_t(s) : kt.knhi - uint32_t(s - kt.nP);
}

// Logical positions of the key order: dense slots 0..nP-1, then the small
// magnitudes as one block (position nP), then dense slots nP..nP+nN-1
// (positions nP+1..).  Count and mass of one position.
__device__ __forceinline__ void kt_position(const KeyTable& kt, int pos, uint32_t sp_count, uint64_t sp_mass,
                                            uint32_t* c, uint64_t* w) {
  if (pos == kt.nP) {
    *c = sp_count;
    *w = sp_mass;
    return;
  }
  const int s = pos < kt.nP ? pos : pos - 1;
  *c = kt.cnt[s];
  *w = uint64_t(kt.cnt[s]) * kt.mass[s];
}

// The first position where the running count (kMass false: reaches `need`)
// or the running mass (kMass true: reaches the top-p target) is reached, in
// every thread, with the count and mass before it.  Each thread covers `spt`
// consecutive positions; (pc, pw) are its exclusive prefixes over the CTA.
template <bool kMass>
__device__ __forceinline__ int kt_locate(KeyTable& kt, int npos, int spt, uint32_t pc, uint64_t pw, uint32_t tc,
                                         uint64_t tw, uint32_t need, const MassTarget& target, uint32_t sp_count,
                                         uint64_t sp_mass, uint32_t* c_before, uint64_t* w_before) {
  const int tid = threadIdx.x;
  if (tid == 0) kt.bc32[0] = 0xFFFFFFFFu;
  cta_sync();
  const bool reach_end = kMass ? (target.trivial || mass_reaches(pw + tw, target)) : (pc + tc >= need);
  const bool reach_start = kMass ? (target.trivial || mass_reaches(pw, target)) : (pc >= need);
  if (reach_end && !reach_start && tc + tw > 0) {   // exactly one thread
    uint32_t c = pc;
    uint64_t w = pw;
    for (int pos = tid * spt; pos < min(npos, (tid + 1) * spt); ++pos) {
      uint32_t pcnt;
      uint64_t pm;
      kt_position(kt, pos, sp_count, sp_mass, &pcnt, &pm);
      const bool hit = kMass ? (pcnt > 0 && (target.trivial || mass_reaches(w + pm, target))) : (c + pcnt >= need);
      if (hit) {
        kt.bc32[0] = uint32_t(pos);
        kt.bc32[1] = c;
        kt.bc64[0] = w;
        break;
      }
      c += pcnt;
      w += pm;
    }
  }
  cta_sync();
  const int pos = int(kt.bc32[0]);
  *c_before = kt.bc32[1];
  *w_before = kt.bc64[0];
  cta_sync();
  return pos;
}

// One row of the general path (see the top of this file).  Returns false,
// having written nothing, when the row needs the per-element path.
template <typename Xf = NoPrep>
__device__ bool key_table_row(KeyTable& kt, const FloatPair* table, const SampleArgs& a, int b,
                              const smp_row_params& prm, const Xf& xf = Xf()) {
  using Vo = VecOps<uint16_t>;
  constexpr int kPer = Vo::kPer;
  const int tid = threadIdx.x, lane = tid & 31;
  const int V = a.vocab;
  if (row_is_greedy(prm) || !sampling_params_valid(prm)) return false;
  const uint16_t* row = reinterpret_cast<const uint16_t*>(a.logits) + size_t(b) * V;
  const uintptr_t r0 = reinterpret_cast<uintptr_t>(row);
  const uintptr_t a0 = (r0 + 15) & ~uintptr_t(15), a1 = (r0 + size_t(V) * 2) & ~uintptr_t(15);
  const bool mid = a1 > a0;
  const int head = mid ? int((a0 - r0) / 2) : V;
  const int tail0 = mid ? int((a1 - r0) / 2) : V;
  const int nvec = mid ? int((a1 - a0) / 16) : 0;
  const uint4* vp = reinterpret_cast<const uint4*>(a0);

  // ---------------- pass 1: the maximum and the per-key counts
  for (int i = tid; i < kKtSlots; i += kThreads) kt.cnt[i] = 0;
  if (tid == 0) {
    kt.sp_n = 0;
    kt.overflow = 0;
  }
  // the first round's vectors (coalesced: thread t takes t + 256 u) give the
  // window's anchor
  uint4 x[kKtU];
  float tmax = -INFINITY;
#pragma unroll
  for (int u = 0; u < kKtU; ++u) {
    const int v = tid + u * kThreads;
    x[u] = v < nvec ? __ldg(vp + v) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  }
  float ze = -INFINITY;   // this thread's edge element (ids before and after the aligned middle)
  int ie = -1;
  if (tid < 16 && tid < head) ie = tid;
  else if (tid >= 16 && tid < 32 && tail0 + tid - 16 < V) ie = tail0 + tid - 16;
  if (ie >= 0) ze = xf(ie, Elem<uint16_t>::widen(row[ie]));
#pragma unroll
  for (int u = 0; u < kKtU; ++u)
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int v = tid + u * kThreads;
      if (v < nvec) tmax = fmaxf(tmax, xf(head + v * kPer + q, Vo::elem(x[u], q)));
    }
  tmax = fmaxf(tmax, ze);
  const float m0 = block_max_f(tmax, kt.redf);
  if (!isfinite(m0)) return false;   // (an error row, or no finite value in the first round)
  if (tid == 0 && !kt_window(kt, m0, prm.temperature)) kt.overflow = 1;
  cta_sync();
  if (kt.overflow) return false;
  bool over = false;
  for (int i = tid; i < 32; i += kThreads) {
    kt.cnt[kKtSlots + i] = 0;
    kt.mass[kKtSlots + i] = 0;
  }
  const uint32_t w_top = kt.kt, w_nhi = kt.knhi, w_np = uint32_t(kt.nP), w_nn = uint32_t(kt.nN), w_kb = kt.kb;
  // one token: its counter (a dummy outside the dense part); the rare small
  // magnitudes and values above the window apart
  auto count = [&](uint32_t id, uint32_t key) {
    const uint32_t s = kt_slot_nb(w_top, w_nhi, w_np, w_nn, key, uint32_t(lane));
    atomicAdd(&kt.cnt[s], 1u);
    if (s >= uint32_t(kKtSlots) && key >= w_kb) {
      if (key > w_top) {
        over = true;
      } else {
        const uint32_t slot = atomicAdd(&kt.sp_n, 1u);
        if (slot < uint32_t(kKtSparse)) kt.sparse[slot] = (uint64_t(key) << 32) | id;
      }
    }
  };
  if (ie >= 0) count(uint32_t(ie), key16_of(ze));
  for (int base = 0;; base += kThreads * kKtU) {
#pragma unroll
    for (int u = 0; u < kKtU; ++u) {
      const int v = base + tid + u * kThreads;
      if (v < nvec) {
        const uint32_t w4[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll 1
        for (int q = 0; q < kPer; ++q) {
          const int id = head + v * kPer + q;
          const uint32_t wq = q < 2 ? w4[0] : q < 4 ? w4[1] : q < 6 ? w4[2] : w4[3];
          const uint32_t h = (q & 1) ? (wq >> 16) : (wq & 0xFFFFu);
          uint32_t key;
          if constexpr (std::is_same<Xf, NoPrep>::value) {
            key = kt_key_bits(h);
          } else {
            const float z = xf(id, __uint_as_float(h << 16));
            tmax = fmaxf(tmax, z);
            key = key16_of(z);
          }
          count(uint32_t(id), key);
        }
        if constexpr (std::is_same<Xf, NoPrep>::value) tmax = fmaxf(tmax, Vo::finish(Vo::vmax(x[u])));
      }
    }
    if (base + kThreads * kKtU >= nvec) break;
#pragma unroll
    for (int u = 0; u < kKtU; ++u) {
      const int v = base + kThreads * kKtU + tid + u * kThreads;
      x[u] = v < nvec ? __ldg(vp + v) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
  }
  if (over) kt.overflow = 1;
  const float m = block_max_f(tmax, kt.redf);   // (its barriers also complete the counts)
  if (kt.overflow || kt.sp_n > uint32_t(kKtSparse) || !isfinite(m)) return false;

  // ---------------- table: E of every key that occurs, and Z
  const RowScale rs = make_row_scale(m, prm.temperature);
  const int nslots = kt.nP + kt.nN;
  const uint32_t sp_n = kt.sp_n;
  for (int s = tid; s < nslots; s += kThreads)
    kt.mass[s] = kt.cnt[s] ? mass_fixed(key_value<uint16_t>(kt_key_of_slot(kt, s)), rs, table) : 0ull;
  uint64_t spm = 0;
  for (int j = tid; j < int(sp_n); j += kThreads) {
    const uint64_t e = mass_fixed(key_value<uint16_t>(uint32_t(kt.sparse[j] >> 32)), rs, table);
    kt.sparse_mass[j] = e;
    spm += e;
  }
  spm = warp_sum<uint64_t>(spm);
  if (lane == 0) kt.scan64[tid >> 5] = spm;
  cta_sync();
  uint64_t sp_mass = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) sp_mass += kt.scan64[w];
  cta_sync();
  // per-thread runs of positions, their counts and masses, scanned
  const int npos = nslots + 1;
  const int spt = (npos + kThreads - 1) / kThreads;
  uint32_t tc = 0;
  uint64_t tw = 0;
  for (int pos = tid * spt; pos < min(npos, (tid + 1) * spt); ++pos) {
    uint32_t c;
    uint64_t w;
    kt_position(kt, pos, sp_n, sp_mass, &c, &w);
    tc += c;
    tw += w;
  }
  uint32_t total_c;
  uint64_t z_total;
  const uint32_t pc = gen_scan<uint32_t>(tc, kt.scan32, &total_c);
  const uint64_t pw = gen_scan<uint64_t>(tw, reinterpret_cast<uint64_t*>(kt.scan64), &z_total);

  // ---------------- select: the shortest of the enabled prefixes
  const bool topk = prm.top_k > 0 && prm.top_k < V;
  const bool topp = prm.top_p < 1.0f;
  const bool minp = prm.min_p > 0.0f && prm.min_p < 1.0f;
  uint64_t len = uint64_t(V);
  // the boundary: keys above `cut` are kept, and the first `n_cut` tokens
  // (id order) of key `cut`; e_cut is their mass, z_kept the kept mass
  uint32_t cut = 0, n_cut = 0;
  uint64_t e_cut = 0, z_kept = z_total;
  bool cut_set = false;
  auto boundary = [&](int pos, uint32_t c_before, uint64_t w_before, uint32_t n) -> bool {
    if (pos == kt.nP) return false;   // the boundary lies among the small magnitudes
    const int s = pos < kt.nP ? pos : pos - 1;
    cut = kt_key_of_slot(kt, s);
    n_cut = n;
    e_cut = kt.mass[s];
    z_kept = w_before + uint64_t(n) * e_cut;
    len = uint64_t(c_before) + n;
    cut_set = true;
    return true;
  };
  const MassTarget none{};
  if (minp) {
    const uint32_t kthr = minp_threshold_key<uint16_t>(kt.bc32, table, rs, prm.temperature, prm.min_p,
                                                       key16_of(m));
    // every token of a key >= kthr is kept: the boundary is kthr's position
    const int s = kt_slot(kt, kthr);
    if (s < 0) return false;   // a threshold among the small magnitudes
    const int pos = s < kt.nP ? s : s + 1;
    // count and mass before `pos`: the thread holding it walks its run
    if (tid == 0) {
      kt.bc32[2] = 0;
      kt.bc64[1] = 0;
    }
    cta_sync();
    if (pos >= tid * spt && pos < (tid + 1) * spt) {
      uint32_t c = pc;
      uint64_t w = pw;
      for (int q = tid * spt; q < pos; ++q) {
        uint32_t qc;
        uint64_t qw;
        kt_position(kt, q, sp_n, sp_mass, &qc, &qw);
        c += qc;
        w += qw;
      }
      kt.bc32[2] = c;
      kt.bc64[1] = w;
    }
    cta_sync();
    const uint32_t cbm = kt.bc32[2];
    const uint64_t wbm = kt.bc64[1];
    cta_sync();
    if (uint64_t(cbm) + kt.cnt[s] < len) boundary(pos, cbm, wbm, kt.cnt[s]);
  }
  if (topk && uint64_t(prm.top_k) < len) {
    if (uint32_t(prm.top_k) > total_c) {
      // the k-th token lies below the window (zero mass): every token of
      // nonzero mass is kept
      len = uint64_t(prm.top_k);
      cut_set = false;
      z_kept = z_total;
    } else {
      uint32_t cb;
      uint64_t wb;
      const int pos = kt_locate<false>(kt, npos, spt, pc, pw, tc, tw, uint32_t(prm.top_k), none, sp_n, sp_mass, &cb,
                                       &wb);
      if (!boundary(pos, cb, wb, uint32_t(prm.top_k) - cb)) return false;
    }
  }
  if (topp) {
    const MassTarget target = make_mass_target(prm.top_p, z_total);
    uint32_t cb;
    uint64_t wb;
    const int pos = kt_locate<true>(kt, npos, spt, pc, pw, tc, tw, 0, target, sp_n, sp_mass, &cb, &wb);
    if (pos == kt.nP) return false;
    const int s = pos < kt.nP ? pos : pos - 1;
    // the crossing inside the key's tokens: the smallest n >= 1 with
    // (mass before + n E) * 2^sh >= top_p * Z (all of them at most)
    const uint64_t e = kt.mass[s];
    uint32_t n = kt.cnt[s];
    if (!target.trivial && e > 0) {
      const u128 have = u128(wb) << target.sh;
      n = 1;
      if (target.rhs > have) {
        const u128 need = target.rhs - have;
        const u128 step = u128(e) << target.sh;
        const u128 q = (need + step - 1) / step;
        n = q > u128(kt.cnt[s]) ? kt.cnt[s] : uint32_t(q);
        if (n == 0) n = 1;
      }
    } else {
      n = 1;
    }
    if (uint64_t(cb) + n < len) boundary(pos, cb, wb, n);
  }
  if (!cut_set) {   // nothing cut among tokens of nonzero mass
    cut = 0;
    n_cut = 0;
    e_cut = 0;
  }

  // ---------------- pass 2: the draw, in token-id order
  // t = floor(u Z_S), u = Philox draw 0 of the row; a token is kept when its
  // key is above `cut`, or equals it and it is among the first n_cut such
  // tokens.  Rounds of kThreads * kKtU vectors, thread t its kKtU consecutive
  // ones; per round each thread's kept mass (the boundary key's tokens
  // counted apart, their rank from the round's scan), a CTA scan, and the
  // thread whose interval holds t walks its ids.
  const uint64_t u53 = uniform53(a.seed, a.offset, a.row_base + uint64_t(b), 0);
  const uint64_t t = uint64_t((u128(u53) * z_kept) >> 53);
  // A token's mass: the table's (the lane's dummy has 0), or, for the rare
  // small magnitudes, the list's.
  auto mass_of_key = [&](uint32_t key, uint32_t id) -> uint64_t {
    const uint32_t s = kt_slot_nb(w_top, w_nhi, w_np, w_nn, key, uint32_t(lane));
    uint64_t e = kt.mass[s];
    if (s >= uint32_t(kKtSlots) && key >= w_kb && key <= w_top)
      for (uint32_t j = 0; j < sp_n; ++j)
        if (uint32_t(kt.sparse[j]) == id) e = kt.sparse_mass[j];
    return e;
  };
  // per token: its kept mass (boundary tokens 0) and whether it is a boundary token
  const uint32_t cut_key = cut_set ? cut : 0u;   // every key is above 0 (-inf's key is 0x007F)
  auto classify_key = [&](uint32_t id, uint32_t key, uint64_t& e, bool& at_cut) {
    at_cut = cut_set && key == cut_key;
    const uint64_t em = mass_of_key(key, id);
    e = key > cut_key ? em : 0ull;
  };
  auto classify = [&](uint32_t id, float z, uint64_t& e, bool& at_cut) { classify_key(id, key16_of(z), e, at_cut); };
  uint64_t run = 0;      // kept mass before this round
  uint32_t run_cut = 0;  // boundary tokens before this round
  int tok = -1;
  if (tid == 0) kt.bc32[4] = 0xFFFFFFFFu;
  // the edges first (ids before the aligned middle), by thread 0, then the
  // middle's rounds, then the ids after it
  if (tid == 0) {
    uint64_t r = 0;
    uint32_t rc = 0;
    for (int i = 0; i < head; ++i) {
      uint64_t e;
      bool ac;
      classify(uint32_t(i), xf(i, Elem<uint16_t>::widen(row[i])), e, ac);
      if (ac) e = rc < n_cut ? e_cut : 0ull, ++rc;
      r += e;
      if (r > t) {
        kt.bc32[4] = uint32_t(i);
        break;
      }
    }
    kt.bc64[2] = r;
    kt.bc32[5] = rc;
  }
  cta_sync();
  tok = int(kt.bc32[4]);
  run = kt.bc64[2];
  run_cut = kt.bc32[5];
  cta_sync();
  for (int base = 0; tok < 0 && base < nvec; base += kThreads * kKtU) {
    const int v0 = base + tid * kKtU;
#pragma unroll
    for (int u = 0; u < kKtU; ++u) x[u] = v0 + u < nvec ? __ldg(vp + v0 + u) : make_uint4(0, 0, 0, 0);
    uint64_t se = 0;
    uint32_t sc = 0;
#pragma unroll
    for (int u = 0; u < kKtU; ++u)
      if (v0 + u < nvec) {
        const uint32_t w4[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll 1
        for (int q = 0; q < kPer; ++q) {
          const int id = head + (v0 + u) * kPer + q;
          const uint32_t wq = q < 2 ? w4[0] : q < 4 ? w4[1] : q < 6 ? w4[2] : w4[3];
          const uint32_t h = (q & 1) ? (wq >> 16) : (wq & 0xFFFFu);
          uint32_t key;
          if constexpr (std::is_same<Xf, NoPrep>::value) key = kt_key_bits(h);
          else key = key16_of(xf(id, __uint_as_float(h << 16)));
          uint64_t e;
          bool ac;
          classify_key(uint32_t(id), key, e, ac);
          se += e;
          sc += ac ? 1u : 0u;
        }
      }
    uint32_t tot_c;
    uint64_t tot_e;
    const uint32_t bc = gen_scan<uint32_t>(sc, kt.scan32, &tot_c);
    const uint64_t be = gen_scan<uint64_t>(se, reinterpret_cast<uint64_t*>(kt.scan64), &tot_e);
    // kept boundary tokens before this thread and in it
    const uint32_t cut_before = run_cut + bc;
    const uint32_t keep_before = min(cut_before, n_cut);
    const uint32_t keep_mine = min(cut_before + sc, n_cut) - keep_before;
    const uint64_t before = run + be + uint64_t(keep_before - min(run_cut, n_cut)) * e_cut;
    const uint64_t mine = se + uint64_t(keep_mine) * e_cut;
    if (mine > 0 && before <= t && t - before < mine) {
      uint64_t r = before;
      uint32_t rc = cut_before;
      bool done = false;
#pragma unroll
      for (int u = 0; u < kKtU; ++u) {
        if (done || v0 + u >= nvec) continue;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
          if (done) continue;
          const int id = head + (v0 + u) * kPer + q;
          uint64_t e;
          bool ac;
          classify(uint32_t(id), xf(id, Vo::elem(x[u], q)), e, ac);
          if (ac) e = rc < n_cut ? e_cut : 0ull, ++rc;
          r += e;
          if (r > t) {
            kt.bc32[4] = uint32_t(id);
            done = true;
          }
        }
      }
    }
    run += tot_e + uint64_t(min(run_cut + tot_c, n_cut) - min(run_cut, n_cut)) * e_cut;
    run_cut += tot_c;
    cta_sync();
    tok = int(kt.bc32[4]);
    cta_sync();
  }
  if (tok < 0 && tid == 0) {
    uint64_t r = run;
    uint32_t rc = run_cut;
    for (int i = tail0; i < V; ++i) {
      uint64_t e;
      bool ac;
      classify(uint32_t(i), xf(i, Elem<uint16_t>::widen(row[i])), e, ac);
      if (ac) e = rc < n_cut ? e_cut : 0ull, ++rc;
      r += e;
      if (r > t) {
        kt.bc32[4] = uint32_t(i);
        break;
      }
    }
  }
  cta_sync();
  tok = int(kt.bc32[4]);

  // ---------------- outputs
  if (tid == 0) {
    a.out_ids[b] = tok;
    if (a.out_probs) {
      const uint64_t e = tok >= 0 ? mass_of_key(key16_of(xf(tok, Elem<uint16_t>::widen(row[tok]))), uint32_t(tok)) : 0;
      a.out_probs[b] = tok >= 0 ? __fdiv_rn(kt_u64_to_f(e), kt_u64_to_f(z_kept)) : __int_as_float(0x7FC00000);
    }
    if (a.kept) a.kept[b] = int32_t(len);
  }
  if (a.full_probs) {
    // p~ of every token (debug); the boundary key's tokens ranked in id order
    const float zf = kt_u64_to_f(z_kept);
    const int warp = tid >> 5;
    if (tid == 0) kt.bc32[6] = 0;
    cta_sync();
    for (int base = 0; base < V; base += kThreads) {
      const int i = base + tid;
      uint64_t e = 0;
      bool ac = false;
      if (i < V) classify(uint32_t(i), xf(i, Elem<uint16_t>::widen(row[i])), e, ac);
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, ac);
      if (lane == 0) kt.scan32[warp] = __popc(bal);
      cta_sync();
      uint32_t before_w = 0, all_w = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (w < warp) before_w += kt.scan32[w];
        all_w += kt.scan32[w];
      }
      const uint32_t rank = kt.bc32[6] + before_w + __popc(bal & ((1u << lane) - 1u));
      if (ac) e = rank < n_cut ? e_cut : 0ull;
      if (i < V) a.full_probs[size_t(b) * V + i] = e ? __fdiv_rn(kt_u64_to_f(e), zf) : 0.0f;
      cta_sync();
      if (tid == 0) kt.bc32[6] += all_w;
      cta_sync();
    }
  }
  cta_sync();
  return true;
}
