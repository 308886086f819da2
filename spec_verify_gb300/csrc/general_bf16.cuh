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
//            in a window that holds every value of nonzero mass, the number
//            of tokens with that value: one counter per value in shared
//            memory.  The window is a run of whole binades (a sign and an
//            exponent: 128 values each) around an early estimate of the
//            maximum; a 512-entry table maps a bf16 pattern's sign and
//            exponent to its binade's first counter, so a token costs a
//            shift, a table load and an atomic add.  Values of very small
//            magnitude (below 2^g, zeros included) would need a counter for
//            every one of their many binades; the few tokens that hold them go
//            to a short list instead (their counters' offsets have bit 15 set,
//            so an OR over a thread's offsets tells it to look for them);
//   table    E(value) = round(exp((z - max z) / T) 2^44) by the double-float
//            exponential for every value that occurs; Z = sum count * E,
//            exact;
//   select   top-k, top-p and min-p on the counters in value order: scans of
//            counts and masses, the crossing found exactly in 128 bits, the
//            number n of tokens of the boundary value that are kept;
//   pass 2   (the row again, normally from L2)  the draw: token ids in order,
//            each token's kept mass looked up in the table (0 past the
//            boundary; a boundary token adds 2^56, which counts it without a
//            branch; the listed tokens' masses from their prefix sums in id
//            order), rounds scanned over the CTA, and the warp of the crossing
//            thread walking its ids.
//
// A row the table cannot take (a value above the window, more small-magnitude
// tokens than the list holds, or a boundary among them) returns false before
// it writes anything, and the caller runs the per-element path instead.
// Included by sample.cu inside namespace smp after general.cuh.
#pragma once

constexpr int kKtBinades = 36;                  // dense binades of the window
constexpr int kKtSlots = kKtBinades * 128;      // one counter per value of a dense binade
constexpr int kKtDummy = kKtSlots;              // 128 counters: binades outside the window
constexpr int kKtAll = kKtSlots + 128;
// Pass 1 counts small-magnitude tokens at byte offsets 32768 + 4 m from the
// counters (over the masses, which are not in use yet): the only offsets with
// bit 15 set.
constexpr uint32_t kKtGapOff = 32768u;
constexpr int kKtSparse = 256;                  // tokens of small magnitude, listed one by one
constexpr int kKtU1 = 4;                        // pass 1: vectors per thread and round (and as many in flight)
constexpr int kKtU2 = 8;                        // pass 2: consecutive vectors per thread and round
constexpr uint64_t kKtCutMark = 1ull << 56;     // pass 2 table entry of the boundary value
constexpr uint32_t kKtFill = 0xFF80FF80u;       // -inf pairs: fill past the row (a binade outside any window)

struct KeyTable {
  uint32_t cnt[kKtAll];
  unsigned long long mass[kKtAll];             // E of the slot's value; in pass 2 the kept mass (or the mark)
  // per (sign, exponent): byte offset of its mantissa-0 counter (pass 1), of
  // its mantissa-0 mass (pass 2: the listed binades' to masses of 0)
  uint32_t lut[512];
  uint32_t gapbits[16];                        // the binades of the list (bit i: lut entry i)
  union {
    struct {
      unsigned long long sparse[kKtSparse];        // (order key << 32) | id of a small-magnitude token
      unsigned long long sparse_mass[kKtSparse];   // its E
    };
    struct {                                       // the same, sorted by id (pass 2)
      uint32_t gid[kKtSparse];
      unsigned long long gpre[kKtSparse + 1];      // exclusive prefix of their kept masses
    };
  };
  unsigned long long scan64[2][kWarps];        // pass 2 rounds: per-warp totals, alternating
  uint32_t scan32[2][kWarps];
  float redf[kWarps];
  uint32_t bc32[8];
  unsigned long long bc64[4];
  uint32_t sp_n;      // small-magnitude tokens seen
  // the window: positive binades with exponents ph, ph-1, .., ph-npb+1 (slots
  // 0 .. 128 npb - 1, mantissa ascending within each), then negative binades
  // with exponents nl .. nl+nnb-1 (slots 128 npb ..); below 2^g the list
  int ph, npb, nl, nnb;
  int pos, neg, pl0, nl0, g;   // the window reaches above / below 0; lowest exponents; the list's bound
  int nsp;            // listed tokens kept in pass 2 (0: none, or not kept)
  uint32_t kb;        // an order key at or below the window's bottom
};
static_assert(sizeof(KeyTable) <= size_t(kBufs) * kBufBytes, "the key table overlays the idle ring");

__device__ __forceinline__ uint32_t key16_of(float z) { return key_of_bits(__float_as_uint(z)) >> 16; }

// The order key of a bf16 bit pattern (-0 as +0, NaN as -inf).
__device__ __forceinline__ uint32_t kt_key_bits(uint32_t h) {
  h = h == 0x8000u ? 0u : h;
  const uint32_t k = (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
  return (h & 0x7FFFu) > 0x7F80u ? 0x007Fu : k;
}

// u64 -> float within two roundings, from 32-bit conversions (the 64-bit
// conversion instructions run on the binary64 pipe, which is narrow on this
// part).
__device__ __forceinline__ float kt_u64_to_f(uint64_t x) {
  return __fmaf_rn(__uint2float_rn(uint32_t(x >> 32)), 0x1p32f, __uint2float_rn(uint32_t(x)));
}

// Byte offset of the counter of bf16 pattern h (its binade's first counter
// plus 4 * mantissa).
__device__ __forceinline__ uint32_t kt_off(const KeyTable& kt, uint32_t h) {
  return kt.lut[h >> 7] + ((h & 0x7Fu) << 2);
}

// Slots and logical positions.  Positions run in descending value order:
// the positive binades (mantissa descending), the small magnitudes as one
// position, the negative binades (magnitude ascending).
__device__ __forceinline__ int kt_pos_of_slot(const KeyTable& kt, int s) {
  return s < kt.npb * 128 ? (s ^ 127) : s + 1;
}
__device__ __forceinline__ int kt_slot_of_pos(const KeyTable& kt, int p) {
  return p < kt.npb * 128 ? (p ^ 127) : p - 1;
}
__device__ __forceinline__ uint32_t kt_bits_of_slot(const KeyTable& kt, int s) {
  if (s < kt.npb * 128) return (uint32_t(kt.ph - (s >> 7)) << 7) | uint32_t(s & 127);
  const int q = s - kt.npb * 128;
  return 0x8000u | (uint32_t(kt.nl + (q >> 7)) << 7) | uint32_t(q & 127);
}

// The window for an estimate m0 of the row maximum (thread 0): every value of
// nonzero mass lies in [m0 - 33 T, max] when the maximum is at most m0 + 8 T
// (checked once it is known): exp((z - max) / T) < 2^-47 below.  Whole
// binades cover it; g, the list's bound, is the smallest exponent that leaves
// at most kKtBinades of them.
__device__ __forceinline__ void kt_window(KeyTable& kt, float m0, float temperature) {
  const float top = fminf(__fmaf_rn(8.0f, temperature, m0), 3.0e38f);
  const float bottom = fmaxf(__fmaf_rn(-33.0f, temperature, m0), -3.0e38f);
  auto ex = [](float x) { return int((__float_as_uint(x) >> 23) & 0xFFu); };
  const bool pos = top > 0.0f, neg = bottom < 0.0f;
  const int ph = pos ? ex(top) : 0;
  const int nh = neg ? ex(bottom) : 0;
  const int pl0 = bottom > 0.0f ? ex(bottom) : 0;   // lowest positive exponent in the window
  const int nl0 = top < 0.0f ? ex(top) : 0;         // lowest negative magnitude exponent in the window
  auto np_of = [&](int g) { return pos ? max(0, ph - max(pl0, g) + 1) : 0; };
  auto nn_of = [&](int g) { return neg ? max(0, nh - max(nl0, g) + 1) : 0; };
  // the binade count does not grow with g, and g = 255 leaves none
  int lo = 0, hi = 255;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (np_of(mid) + nn_of(mid) <= kKtBinades) hi = mid;
    else lo = mid + 1;
  }
  const int g = lo, np = np_of(g), nn = nn_of(g);
  kt.ph = ph;
  kt.npb = np;
  kt.nl = max(nl0, g);
  kt.nnb = nn;
  kt.pos = pos;
  kt.neg = neg;
  kt.pl0 = pl0;
  kt.nl0 = nl0;
  kt.g = g;
  const uint32_t kbot = key16_of(bottom);
  kt.kb = kbot > 0x0080u ? kbot - 1u : 0x0080u;
}

// Binade i = sign * 256 + exponent (after kt_window): its first slot, or -1
// for the list's binades, or kKtDummy outside the window.
__device__ __forceinline__ int kt_binade_slot(const KeyTable& kt, int i) {
  const int s = i >> 8, e = i & 0xFF;
  if (s == 0 && kt.pos && e <= kt.ph && e > kt.ph - kt.npb) return (kt.ph - e) * 128;
  if (s == 1 && kt.neg && e >= kt.nl && e < kt.nl + kt.nnb) return (kt.npb + e - kt.nl) * 128;
  if (e < kt.g && ((s == 0 && kt.pos && e >= kt.pl0) || (s == 1 && kt.neg && e >= kt.nl0))) return -1;
  return kKtDummy;
}

// Pass 1 table entry: byte offset of the binade's first counter.
__device__ __forceinline__ uint32_t kt_lut_entry(const KeyTable& kt, int i) {
  const int s = kt_binade_slot(kt, i);
  return s < 0 ? kKtGapOff : uint32_t(s) * 4u;
}

__device__ __forceinline__ bool kt_listed_binade(const KeyTable& kt, uint32_t h) {
  return (kt.gapbits[h >> 12] >> ((h >> 7) & 31)) & 1u;
}

// A token of a small-magnitude binade in pass 1: listed if not below the window.
__device__ __forceinline__ void kt_list(KeyTable& kt, uint32_t h, uint32_t id) {
  const uint32_t key = kt_key_bits(h);
  if (key >= kt.kb) {
    const uint32_t j = atomicAdd(&kt.sp_n, 1u);
    if (j < uint32_t(kKtSparse)) kt.sparse[j] = (uint64_t(key) << 32) | id;
  }
}

// The first position where the running count (kMass false: reaches `need`)
// or the running mass (kMass true: reaches the top-p target) is reached, in
// every thread, with the count and mass before it.  Each thread covers `spt`
// <= 32 consecutive positions; (pc, pw) are its exclusive prefixes over the
// CTA.  The thread whose run holds the crossing hands it to warp 0, whose
// lanes take one position each.
template <bool kMass>
__device__ __forceinline__ int kt_locate(KeyTable& kt, int npos, int spt, uint32_t pc, uint64_t pw, uint32_t tc,
                                         uint64_t tw, uint32_t need, const MassTarget& target, uint32_t sp_count,
                                         uint64_t sp_mass, uint32_t* c_before, uint64_t* w_before) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    kt.bc32[4] = 0xFFFFFFFFu;
    kt.bc32[6] = 0xFFFFFFFFu;
  }
  cta_sync();
  const bool reach_end = kMass ? (target.trivial || mass_reaches(pw + tw, target)) : (pc + tc >= need);
  const bool reach_start = kMass ? (target.trivial || mass_reaches(pw, target)) : (pc >= need);
  if (reach_end && !reach_start && tc + tw > 0) {   // exactly one thread
    kt.bc32[4] = uint32_t(tid);
    kt.bc32[5] = pc;
    kt.bc64[0] = pw;
  }
  cta_sync();
  const uint32_t owner = kt.bc32[4];
  if (tid < 32 && owner != 0xFFFFFFFFu) {
    const int lane = tid;
    const int p = int(owner) * spt + lane;
    const bool valid = lane < spt && p < npos;
    uint32_t pcnt = 0;
    uint64_t pm = 0;
    if (valid) {
      if (p == kt.npb * 128) {
        pcnt = sp_count;
        pm = sp_mass;
      } else {
        const int s = kt_slot_of_pos(kt, p);
        pcnt = kt.cnt[s];
        pm = uint64_t(pcnt) * kt.mass[s];
      }
    }
    const uint32_t cb = kt.bc32[5] + warp_inclusive_scan<uint32_t>(pcnt) - pcnt;
    const uint64_t wb = kt.bc64[0] + warp_inclusive_scan<uint64_t>(pm) - pm;
    const bool hit =
        valid && (kMass ? (pcnt > 0 && (target.trivial || mass_reaches(wb + pm, target))) : (cb + pcnt >= need));
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, hit);
    if (bal && lane == __ffs(bal) - 1) {
      kt.bc32[6] = uint32_t(p);
      kt.bc32[7] = cb;
      kt.bc64[1] = wb;
    }
  }
  cta_sync();
  const int pos = int(kt.bc32[6]);
  *c_before = kt.bc32[7];
  *w_before = kt.bc64[1];
  cta_sync();
  return pos;
}

// The smallest n in [1, cnt] with ((w + n e) << sh) >= rhs, or cnt: a float
// estimate of the quotient, corrected by exact products (n < 2^31).
__device__ __forceinline__ uint32_t kt_tokens_to_reach(uint64_t w, uint64_t e, uint32_t cnt, const MassTarget& t) {
  if (t.trivial || e == 0) return 1;
  const u128 have = u128(w) << t.sh;
  if (t.rhs <= have) return 1;
  const u128 need = t.rhs - have;
  const u128 step = u128(e) << t.sh;
  auto to_f = [](u128 x) { return __fmaf_rn(kt_u64_to_f(uint64_t(x >> 64)), 0x1p64f, kt_u64_to_f(uint64_t(x))); };
  float qf = ceilf(__fdiv_rn(to_f(need), to_f(step)));
  qf = fminf(fmaxf(qf, 1.0f), float(cnt));
  uint32_t q = uint32_t(qf);
  while (q < cnt && u128(q) * step < need) ++q;
  while (q > 1 && u128(q - 1) * step >= need) --q;
  return q;
}

// One row of the general path (see the top of this file).  Returns false,
// having written nothing, when the row needs the per-element path.
template <typename Xf = NoPrep>
__device__ bool key_table_row(KeyTable& kt, const FloatPair* table, const SampleArgs& a, int b,
                              const smp_row_params& prm, const Xf& xf = Xf()) {
  using Vo = VecOps<uint16_t>;
  constexpr int kPer = Vo::kPer;
  constexpr bool kRaw = std::is_same<Xf, NoPrep>::value;
  const int tid = threadIdx.x;
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
  unsigned char* const cntb = reinterpret_cast<unsigned char*>(kt.cnt);
  const unsigned char* const massb = reinterpret_cast<const unsigned char*>(kt.mass);
  // the bf16 pattern of element q of a vector, after the row's transform
  auto pattern = [&](const uint4& x, int q, int id) -> uint32_t {
    if constexpr (kRaw) {
      const uint32_t w = q < 2 ? x.x : q < 4 ? x.y : q < 6 ? x.z : x.w;
      return (q & 1) ? (w >> 16) : (w & 0xFFFFu);
    } else {
      return __float_as_uint(xf(id, Vo::elem(x, q))) >> 16;
    }
  };
  // a raw bf16 pattern of token id, after the row's transform
  auto transform = [&](uint32_t h, uint32_t id) -> uint32_t {
    if constexpr (kRaw) return h;
    else return __float_as_uint(xf(int(id), __uint_as_float(h << 16))) >> 16;
  };
  auto edge_pattern = [&](int i) -> uint32_t {
    if constexpr (kRaw) return uint32_t(row[i]);
    else return __float_as_uint(xf(i, Elem<uint16_t>::widen(row[i]))) >> 16;
  };

  // ---------------- pass 1: the maximum and the per-value counts
  // the first round's vectors (coalesced: thread t takes t + 256 u) give the
  // window's anchor; the counters are cleared while they load
  uint4 x[kKtU1];
#pragma unroll
  for (int u = 0; u < kKtU1; ++u) {
    const int v = tid + u * kThreads;
    x[u] = v < nvec ? __ldg(vp + v) : make_uint4(kKtFill, kKtFill, kKtFill, kKtFill);
  }
  for (int i = tid; i < kKtAll; i += kThreads) kt.cnt[i] = 0;
  if (tid == 0) kt.sp_n = 0;
  uint32_t he = kKtFill & 0xFFFFu;   // this thread's edge element (ids before and after the aligned middle)
  int ie = -1;
  if (tid < 16 && tid < head) ie = tid;
  else if (tid >= 16 && tid < 32 && tail0 + tid - 16 < V) ie = tail0 + tid - 16;
  if (ie >= 0) he = edge_pattern(ie);
  float tmax = __uint_as_float(he << 16);
  uint32_t vmax2 = Vo::neg_inf();   // raw rows: the running maximum of bf16 pairs
#pragma unroll
  for (int u = 0; u < kKtU1; ++u) {
    if constexpr (kRaw) {
      vmax2 = Vo::max2(vmax2, Vo::vmax(x[u]));
    } else {
      const int v = tid + u * kThreads;
#pragma unroll
      for (int q = 0; q < kPer; ++q)
        if (v < nvec) tmax = fmaxf(tmax, __uint_as_float(pattern(x[u], q, head + v * kPer + q) << 16));
    }
  }
  if constexpr (kRaw) tmax = fmaxf(tmax, Vo::finish(vmax2));
  const float m0 = block_max_f(tmax, kt.redf);
  if (!isfinite(m0)) return false;   // (an error row, or no finite value in the first round)
  if (tid == 0) kt_window(kt, m0, prm.temperature);
  cta_sync();
  for (int i = tid; i < 512; i += kThreads) kt.lut[i] = kt_lut_entry(kt, i);
  cta_sync();

  // one token: its counter; a small-magnitude one also to the list
  auto count = [&](uint32_t h, uint32_t id) {
    const uint32_t off = kt_off(kt, h);
    atomicAdd(reinterpret_cast<uint32_t*>(cntb + off), 1u);
    if (off & kKtGapOff) kt_list(kt, h, id);
  };
  if (ie >= 0) count(he, uint32_t(ie));
  for (int base = 0;; base += kThreads * kKtU1) {
    const bool more = base + kThreads * kKtU1 < nvec;
    uint4 y[kKtU1];
#pragma unroll
    for (int u = 0; u < kKtU1; ++u) {   // the next round's vectors, in flight meanwhile
      const int v = base + kThreads * kKtU1 + tid + u * kThreads;
      y[u] = v < nvec ? __ldg(vp + v) : make_uint4(kKtFill, kKtFill, kKtFill, kKtFill);
    }
    if constexpr (kRaw) {
      // pairs of bf16 values; fill vectors past the row count in counters
      // outside the window
      // every offset of the round first, then the atomics: an atomic may not
      // pass a later table load (the compiler cannot tell them apart), so
      // interleaving them would serialise two shared-memory latencies per pair
      uint32_t off[kKtU1 * 8];
#pragma unroll
      for (int u = 0; u < kKtU1; ++u) {
        vmax2 = Vo::max2(vmax2, Vo::vmax(x[u]));
        const uint32_t w4[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t w = w4[k];
          off[u * 8 + 2 * k] = kt.lut[(w >> 7) & 0x1FFu] + ((w & 0x7Fu) << 2);
          off[u * 8 + 2 * k + 1] = kt.lut[w >> 23] + ((w >> 14) & 0x1FCu);
        }
      }
      uint32_t seen = 0;   // OR of the offsets: bit 15 when a listed binade occurred
#pragma unroll
      for (int j = 0; j < kKtU1 * 8; ++j) {
        atomicAdd(reinterpret_cast<uint32_t*>(cntb + off[j]), 1u);
        seen |= off[j];
      }
      if (seen & kKtGapOff) {   // rare: list this round's small magnitudes
        for (int u = 0; u < kKtU1; ++u) {
          const int v = base + tid + u * kThreads;
          if (v >= nvec) break;
          const uint4 xw = __ldg(vp + v);
          for (int q = 0; q < kPer; ++q) {
            const uint32_t h = pattern(xw, q, 0);
            if (kt_off(kt, h) & kKtGapOff) kt_list(kt, h, uint32_t(head + v * kPer + q));
          }
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < kKtU1; ++u) {
        const int v = base + tid + u * kThreads;
        if (v < nvec) {
#pragma unroll
          for (int q = 0; q < kPer; ++q) {
            const int id = head + v * kPer + q;
            const uint32_t h = pattern(x[u], q, id);
            tmax = fmaxf(tmax, __uint_as_float(h << 16));
            count(h, uint32_t(id));
          }
        }
      }
    }
    if (!more) break;
#pragma unroll
    for (int u = 0; u < kKtU1; ++u) x[u] = y[u];
  }
  if constexpr (kRaw) tmax = fmaxf(tmax, Vo::finish(vmax2));
  const float m = block_max_f(tmax, kt.redf);   // (its barriers also complete the counts)
  // the maximum must lie in the window: a binade with counters or the list
  const uint32_t lm = isfinite(m) ? kt.lut[__float_as_uint(m) >> 23] : uint32_t(kKtDummy) * 4u;
  if (lm == uint32_t(kKtDummy) * 4u || kt.sp_n > uint32_t(kKtSparse)) return false;

  // ---------------- table: E of every value that occurs, and Z
  const RowScale rs = make_row_scale(m, prm.temperature);
  const int nslots = (kt.npb + kt.nnb) * 128;
  const uint32_t sp_n = kt.sp_n;
  // (four slots per thread and step: four independent exponentials in flight)
  for (int s0 = tid; s0 < nslots; s0 += 4 * kThreads) {
    uint32_t c[4];
    uint64_t e[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = s0 + j * kThreads < nslots ? kt.cnt[s0 + j * kThreads] : 0u;
    if (c[0] | c[1] | c[2] | c[3]) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        e[j] = mass_fixed(__uint_as_float(kt_bits_of_slot(kt, min(s0 + j * kThreads, nslots - 1)) << 16), rs, table);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (s0 + j * kThreads < nslots) kt.mass[s0 + j * kThreads] = c[j] ? e[j] : 0ull;
  }
  for (int s = kKtSlots + tid; s < kKtAll; s += kThreads) kt.mass[s] = 0;
  // the listed tokens: E, and their rank in id order
  uint64_t spe = 0;
  uint32_t sp_id = 0, sp_rank = 0;
  if (tid < int(sp_n)) {
    const uint64_t ent = kt.sparse[tid];
    sp_id = uint32_t(ent);
    spe = mass_fixed(key_value<uint16_t>(uint32_t(ent >> 32)), rs, table);
    for (uint32_t j = 0; j < sp_n; ++j) sp_rank += uint32_t(kt.sparse[j]) < sp_id ? 1u : 0u;
  }
  cta_sync();   // the masses are in place
  // per-thread runs of positions, their counts and masses (the list's
  // position apart), and the list's masses: one CTA scan of the three
  const int gp = kt.npb * 128;
  const int npos = nslots + 1;
  const int spt = (npos + kThreads - 1) / kThreads;
  const int p_lo = tid * spt, p_hi = min(npos, (tid + 1) * spt);
  uint32_t tc = 0;
  uint64_t tw = 0;
#pragma unroll 4
  for (int p = p_lo; p < p_hi; ++p) {
    if (p != gp) {
      const int sl = kt_slot_of_pos(kt, p);
      const uint32_t c = kt.cnt[sl];
      tc += c;
      tw += uint64_t(c) * kt.mass[sl];
    }
  }
  const bool own_gp = gp >= p_lo && gp < p_hi;
  if (own_gp) tc += sp_n;
  const uint32_t ic = warp_inclusive_scan<uint32_t>(tc);
  const uint64_t iw = warp_inclusive_scan<uint64_t>(tw);
  const uint64_t is = warp_inclusive_scan<uint64_t>(spe);
  if ((tid & 31) == 31) {
    kt.scan32[0][tid >> 5] = ic;
    kt.scan64[0][tid >> 5] = iw;
    kt.scan64[1][tid >> 5] = is;
  }
  cta_sync();   // (also: every read of the unsorted list is done)
  uint32_t pc = ic - tc, total_c = 0;
  uint64_t pw = iw - tw, z_total = 0, sp_mass = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    if (w < (tid >> 5)) {
      pc += kt.scan32[0][w];
      pw += kt.scan64[0][w];
    }
    total_c += kt.scan32[0][w];
    z_total += kt.scan64[0][w];
    sp_mass += kt.scan64[1][w];
  }
  // the list's mass sits at position gp
  if (own_gp) tw += sp_mass;
  if (p_lo > gp) pw += sp_mass;
  z_total += sp_mass;
  if (tid < int(sp_n)) {
    kt.gid[sp_rank] = sp_id;
    kt.gpre[sp_rank + 1] = spe;   // prefix sums below, once the masses are in place
  }
  cta_sync();
  // the list's prefix sums, by warp 0
  if (tid < 32) {
    constexpr int kPerLane = kKtSparse / 32;
    uint64_t v[kPerLane], sum = 0;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      const int r = tid * kPerLane + j;
      v[j] = r < int(sp_n) ? kt.gpre[r + 1] : 0ull;
      sum += v[j];
    }
    uint64_t run_l = warp_inclusive_scan<uint64_t>(sum) - sum;
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      const int r = tid * kPerLane + j;
      run_l += v[j];
      if (r < int(sp_n)) kt.gpre[r + 1] = run_l;
    }
    if (tid == 0) kt.gpre[0] = 0;
  }

  // ---------------- select: the shortest of the enabled prefixes
  const bool topk = prm.top_k > 0 && prm.top_k < V;
  const bool topp = prm.top_p < 1.0f;
  const bool minp = prm.min_p > 0.0f && prm.min_p < 1.0f;
  uint64_t len = uint64_t(V);
  // the boundary: positions before pos_cut are kept, and the first n_cut
  // tokens (id order) of the value at pos_cut; e_cut is their mass, z_kept
  // the kept mass
  int pos_cut = npos;
  uint32_t n_cut = 0;
  uint64_t e_cut = 0, z_kept = z_total;
  auto boundary = [&](int pos, uint32_t c_before, uint64_t w_before, uint32_t n) -> bool {
    if (pos == gp) return false;   // the boundary lies among the small magnitudes
    const int s = kt_slot_of_pos(kt, pos);
    pos_cut = pos;
    n_cut = n;
    e_cut = kt.mass[s];
    z_kept = w_before + uint64_t(n) * e_cut;
    len = uint64_t(c_before) + n;
    return true;
  };
  const MassTarget none{};
  if (minp) {
    const uint32_t kthr = minp_threshold_key<uint16_t>(kt.bc32, table, rs, prm.temperature, prm.min_p,
                                                       key16_of(m));
    // every token of a value >= the threshold is kept: the boundary is its
    // position (a threshold outside the counters: the per-element path)
    const uint32_t hthr = (kthr & 0x8000u) ? (kthr & 0x7FFFu) : (~kthr & 0xFFFFu);
    const uint32_t off = kt_off(kt, hthr);
    if (off >= uint32_t(kKtSlots) * 4u || (hthr & 0x7FFFu) == 0) return false;
    const int s = int(off >> 2);
    const int pos = kt_pos_of_slot(kt, s);
    // count and mass before `pos`: the thread holding it walks its run
    if (tid == 0) {
      kt.bc32[6] = 0;
      kt.bc64[1] = 0;
    }
    cta_sync();
    if (pos >= tid * spt && pos < (tid + 1) * spt) {
      uint32_t c = pc;
      uint64_t w = pw;
      for (int p = tid * spt; p < pos; ++p) {
        if (p == gp) {
          c += sp_n;
          w += sp_mass;
        } else {
          const int q = kt_slot_of_pos(kt, p);
          c += kt.cnt[q];
          w += uint64_t(kt.cnt[q]) * kt.mass[q];
        }
      }
      kt.bc32[6] = c;
      kt.bc64[1] = w;
    }
    cta_sync();
    const uint32_t cbm = kt.bc32[6];
    const uint64_t wbm = kt.bc64[1];
    cta_sync();
    if (uint64_t(cbm) + kt.cnt[s] < len) boundary(pos, cbm, wbm, kt.cnt[s]);
  }
  if (topk && uint64_t(prm.top_k) < len) {
    if (uint32_t(prm.top_k) > total_c) {
      // the k-th token lies below the window (zero mass): every token of
      // nonzero mass is kept
      len = uint64_t(prm.top_k);
      pos_cut = npos;
      n_cut = 0;
      z_kept = z_total;
    } else {
      uint32_t cb;
      uint64_t wb;
      const int pos = kt_locate<false>(kt, npos, spt, pc, pw, tc, tw, uint32_t(prm.top_k), none, sp_n, sp_mass, &cb,
                                       &wb);
      if (pos < 0 || !boundary(pos, cb, wb, uint32_t(prm.top_k) - cb)) return false;
    }
  }
  if (topp) {
    const MassTarget target = make_mass_target(prm.top_p, z_total);
    uint32_t cb;
    uint64_t wb;
    const int pos = kt_locate<true>(kt, npos, spt, pc, pw, tc, tw, 0, target, sp_n, sp_mass, &cb, &wb);
    if (pos < 0 || pos == gp) return false;
    const int s = kt_slot_of_pos(kt, pos);
    // the crossing inside the value's tokens: the smallest n >= 1 with
    // (mass before + n E) * 2^sh >= top_p * Z (all of them at most)
    const uint32_t n = kt_tokens_to_reach(wb, kt.mass[s], kt.cnt[s], target);
    if (uint64_t(cb) + n < len) boundary(pos, cb, wb, n);
  }
  const bool gap_kept = pos_cut > gp && sp_n > 0;   // the listed tokens are kept (all or none)
  // the pass 2 tables: kept E before the boundary, the mark at it, 0 after;
  // each binade's first mass (the list's binades and the rest: masses of 0)
  cta_sync();
  if (pos_cut < npos)
    for (int s = tid; s < nslots; s += kThreads) {
      const int p = kt_pos_of_slot(kt, s);
      if (p >= pos_cut) kt.mass[s] = p == pos_cut ? kKtCutMark : 0ull;
    }
  for (int i = tid; i < 512; i += kThreads) {
    const int s = kt_binade_slot(kt, i);
    kt.lut[i] = uint32_t(s < 0 ? kKtDummy : s) * 8u;
    const uint32_t bits = __ballot_sync(0xFFFFFFFFu, s < 0);
    if ((tid & 31) == 0) kt.gapbits[i >> 5] = bits;
  }
  cta_sync();

  // ---------------- pass 2: the draw, in token-id order
  // t = floor(u Z_S), u = Philox draw 0 of the row; the token is the first
  // kept one (id order) whose running mass passes t; a token is kept when its
  // value comes before the boundary, or is the boundary value and it is among
  // the first n_cut such tokens.  Rounds of kThreads * kKtU2 vectors, thread t
  // its kKtU2 consecutive ones; per round each thread's kept mass (the
  // boundary tokens counted in bits 56.., their rank from the round's scan),
  // a CTA scan, and the warp of the thread whose interval holds t walks its
  // ids.
  const uint64_t u53 = uniform53(a.seed, a.offset, a.row_base + uint64_t(b), 0);
  const uint64_t t = uint64_t((u128(u53) * z_kept) >> 53);
  const int nsp = gap_kept ? int(sp_n) : 0;
  // listed ids below x, and their kept mass
  auto listed_below = [&](uint32_t x) -> int {
    int lo = 0, hi = nsp;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (kt.gid[mid] < x) lo = mid + 1;
      else hi = mid;
    }
    return lo;
  };
  auto listed_mass = [&](uint32_t id) -> uint64_t {
    const int r = listed_below(id);
    return r < nsp && kt.gid[r] == id ? kt.gpre[r + 1] - kt.gpre[r] : 0ull;
  };
  auto mass_at = [&](uint32_t off) -> uint64_t {
    return *reinterpret_cast<const unsigned long long*>(massb + off);
  };
  // a token's pass 2 entry: kept E, the mark, or 0
  auto entry = [&](uint32_t h, uint32_t id) -> uint64_t {
    if (kt_listed_binade(kt, h)) return listed_mass(id);
    return mass_at(kt.lut[h >> 7] + ((h & 0x7Fu) << 3));
  };
  // The walk runs from whichever end of the row is nearer the draw.  Walking
  // backwards is the forward walk over the reversed ids with
  // t_b = Z_S - 1 - t: the token is the first (reversed) whose running mass
  // passes t_b, and of the boundary value's tokens the last n_cut (id order)
  // are kept.  kept(r): boundary tokens kept among the first r in walk order.
  const bool bwd = t >= z_kept - t;
  const uint64_t t_walk = bwd ? z_kept - 1 - t : t;
  const uint32_t cnt_cut = pos_cut < npos ? kt.cnt[kt_slot_of_pos(kt, pos_cut)] : 0u;
  const uint32_t skip = cnt_cut - n_cut;
  auto kept = [&](uint32_t r) -> uint32_t { return bwd ? (r > skip ? r - skip : 0u) : min(r, n_cut); };
  // walking: the running mass r and boundary count rc over one token
  auto step = [&](uint64_t ent, uint64_t& r, uint32_t& rc) {
    if (ent == kKtCutMark) {
      r += kept(rc + 1) > kept(rc) ? e_cut : 0ull;
      ++rc;
    } else {
      r += ent;
    }
  };
  // the row's edges in walk order (ids before and after the aligned middle)
  auto walk_edge = [&](bool first, uint64_t& r, uint32_t& rc) -> int {
    const bool lead = first != bwd;   // the head walked forwards, or the tail backwards
    const int n = lead ? head : V - tail0;
    for (int j = 0; j < n; ++j) {
      const int i = lead ? (bwd ? head - 1 - j : j) : (bwd ? V - 1 - j : tail0 + j);
      step(entry(edge_pattern(i), uint32_t(i)), r, rc);
      if (r > t_walk) return i;
    }
    return -1;
  };
  uint64_t run = 0;      // kept mass before this round (walk order)
  uint32_t run_cut = 0;  // boundary tokens before this round
  int tok = -1;
  if (tid == 0) {
    uint64_t r = 0;
    uint32_t rc = 0;
    kt.bc32[4] = uint32_t(walk_edge(true, r, rc));
    kt.bc64[2] = r;
    kt.bc32[5] = rc;
  }
  cta_sync();
  tok = int(kt.bc32[4]);
  run = kt.bc64[2];
  run_cut = kt.bc32[5];
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int kRound = kThreads * kKtU2;
  for (int base = 0, rnd = 0; tok < 0 && base < nvec; base += kRound, rnd ^= 1) {
    // this thread's kKtU2 vectors: the tid-th chunk of the round in walk order
    const int v0 = bwd ? nvec - base - (tid + 1) * kKtU2 : base + tid * kKtU2;
    uint4 xv[kKtU2];
#pragma unroll
    for (int u = 0; u < kKtU2; ++u)
      xv[u] = v0 + u >= 0 && v0 + u < nvec ? __ldg(vp + v0 + u) : make_uint4(kKtFill, kKtFill, kKtFill, kKtFill);
    uint64_t se = 0;
    if constexpr (kRaw) {
#pragma unroll
      for (int u = 0; u < kKtU2; ++u) {
        const uint32_t w4[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t w = w4[k];
          const uint32_t o0 = kt.lut[(w >> 7) & 0x1FFu] + ((w & 0x7Fu) << 3);
          const uint32_t o1 = kt.lut[w >> 23] + ((w >> 13) & 0x3F8u);
          se += mass_at(o0) + mass_at(o1);
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < kKtU2; ++u)
        if (v0 + u >= 0 && v0 + u < nvec) {
          const uint32_t id0 = uint32_t(head + (v0 + u) * kPer);
#pragma unroll
          for (int q = 0; q < kPer; ++q) {
            const uint32_t h = pattern(xv[u], q, int(id0) + q);
            se += kt_listed_binade(kt, h) ? 0ull : mass_at(kt.lut[h >> 7] + ((h & 0x7Fu) << 3));
          }
        }
    }
    const int va = max(v0, 0), vb = min(v0 + kKtU2, nvec);
    if (nsp > 0 && va < vb) {   // the listed tokens among this thread's ids
      const uint32_t lo = uint32_t(head + va * kPer), hi = uint32_t(head + vb * kPer);
      se += kt.gpre[listed_below(hi)] - kt.gpre[listed_below(lo)];
    }
    const uint32_t sc = uint32_t(se >> 56);
    se &= kKtCutMark - 1;
    // one barrier per round: warp totals alternate between two buffers
    const uint32_t ic = warp_inclusive_scan<uint32_t>(sc);
    const uint64_t ie64 = warp_inclusive_scan<uint64_t>(se);
    if (lane == 31) {
      kt.scan32[rnd][warp] = ic;
      kt.scan64[rnd][warp] = ie64;
    }
    cta_sync();
    uint32_t bc = ic - sc, tot_c = 0;
    uint64_t be = ie64 - se, tot_e = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t wc = kt.scan32[rnd][w];
      const uint64_t we = kt.scan64[rnd][w];
      if (w < warp) {
        bc += wc;
        be += we;
      }
      tot_c += wc;
      tot_e += we;
    }
    const uint64_t round_mass = tot_e + uint64_t(kept(run_cut + tot_c) - kept(run_cut)) * e_cut;
    if (run + round_mass > t_walk) {   // the draw falls in this round (every thread alike)
      // kept boundary tokens before this thread and in it
      const uint32_t cut_before = run_cut + bc;
      const uint64_t before = run + be + uint64_t(kept(cut_before) - kept(run_cut)) * e_cut;
      const uint64_t mine = se + uint64_t(kept(cut_before + sc) - kept(cut_before)) * e_cut;
      const uint32_t hit = __ballot_sync(0xFFFFFFFFu, mine > 0 && before <= t_walk && t_walk - before < mine);
      if (hit) {
        // this warp walks the crossing thread's ids: lane l the l-th pair in
        // walk order (backwards: the pairs from the last, high id first)
        const int src = __ffs(hit) - 1;
        const int cv0 = __shfl_sync(0xFFFFFFFFu, v0, src);
        const uint64_t cb = shfl_u64(before, src);
        const uint32_t ccut = __shfl_sync(0xFFFFFFFFu, cut_before, src);
        const int pr = bwd ? 31 - lane : lane;
        const int v = cv0 + (pr >> 2);
        const bool valid = v >= 0 && v < nvec;
        const uint32_t w = valid ? __ldg(reinterpret_cast<const uint32_t*>(vp + v) + (pr & 3)) : kKtFill;
        const uint32_t id_lo = uint32_t(head + v * kPer + 2 * (pr & 3));
        const uint32_t id0 = bwd ? id_lo + 1 : id_lo, id1 = bwd ? id_lo : id_lo + 1;
        const uint32_t h0 = bwd ? (w >> 16) : (w & 0xFFFFu), h1 = bwd ? (w & 0xFFFFu) : (w >> 16);
        const uint64_t e0 = valid ? entry(transform(h0, id0), id0) : 0ull;
        const uint64_t e1 = valid ? entry(transform(h1, id1), id1) : 0ull;
        const uint32_t c0 = e0 == kKtCutMark, c1 = e1 == kKtCutMark;
        const uint32_t rank0 = ccut + warp_inclusive_scan<uint32_t>(c0 + c1) - (c0 + c1);
        const uint64_t m0 = c0 ? (kept(rank0 + 1) > kept(rank0) ? e_cut : 0ull) : e0;
        const uint64_t m1 = c1 ? (kept(rank0 + c0 + 1) > kept(rank0 + c0) ? e_cut : 0ull) : e1;
        const uint64_t r0 = cb + warp_inclusive_scan<uint64_t>(m0 + m1) - m1;
        const uint64_t r1 = r0 + m1;
        const uint32_t found = __ballot_sync(0xFFFFFFFFu, r1 > t_walk);
        if (found && lane == __ffs(found) - 1) kt.bc32[4] = r0 > t_walk ? id0 : id1;
      }
      cta_sync();
      tok = int(kt.bc32[4]);
      break;
    }
    run += round_mass;
    run_cut += tot_c;
  }
  if (tok < 0 && tid == 0) {
    uint64_t r = run;
    uint32_t rc = run_cut;
    kt.bc32[4] = uint32_t(walk_edge(false, r, rc));
  }
  cta_sync();
  tok = int(kt.bc32[4]);

  // ---------------- outputs
  if (tid == 0) {
    a.out_ids[b] = tok;
    if (a.out_probs) {
      uint64_t e = 0;
      if (tok >= 0) {
        const uint64_t ent = entry(edge_pattern(tok), uint32_t(tok));
        e = ent == kKtCutMark ? e_cut : ent;
      }
      a.out_probs[b] = tok >= 0 ? __fdiv_rn(kt_u64_to_f(e), kt_u64_to_f(z_kept)) : __int_as_float(0x7FC00000);
    }
    if (a.kept) a.kept[b] = int32_t(len);
  }
  if (a.full_probs) {
    // p~ of every token (debug); the boundary value's tokens ranked in id order
    const float zf = kt_u64_to_f(z_kept);
    if (tid == 0) kt.bc32[6] = 0;
    cta_sync();
    for (int base = 0; base < V; base += kThreads) {
      const int i = base + tid;
      const uint64_t ent = i < V ? entry(edge_pattern(i), uint32_t(i)) : 0ull;
      const bool ac = ent == kKtCutMark;
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, ac);
      if (lane == 0) kt.scan32[0][warp] = __popc(bal);
      cta_sync();
      uint32_t before_w = 0, all_w = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        if (w < warp) before_w += kt.scan32[0][w];
        all_w += kt.scan32[0][w];
      }
      const uint32_t rank = kt.bc32[6] + before_w + __popc(bal & ((1u << lane) - 1u));
      const uint64_t e = ac ? (rank < n_cut ? e_cut : 0ull) : ent;
      if (i < V) a.full_probs[size_t(b) * V + i] = e ? __fdiv_rn(kt_u64_to_f(e), zf) : 0.0f;
      cta_sync();
      if (tid == 0) kt.bc32[6] += all_w;
      cta_sync();
    }
  }
  cta_sync();
  return true;
}
