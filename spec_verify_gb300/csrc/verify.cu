// Speculative-decoding verifier ("Decoding & Speculative Sampling", section
// 39.4, eqs. 39.3 and 39.4; "Speculative decoding -- Hinglish notes", section
// "The Algorithm (Step-by-Step)"; "Efficient Inference & Compression", section
// "Speculative decoding").
//
// Two kernels on the caller's stream:
//   verify_pos_kernel      one CTA per logit row (b, position, target or
//                          draft): the row maximum, the fixed-point mass Z
//                          and the draft token's mass, written to the
//                          workspace;
//   verify_resolve_kernel  one cluster per batch row: the accept tests in
//                          order, then the replacement draw from
//                          max(0, p_j - q_j) at the first rejection j, or the
//                          bonus draw from p_K.
// Per-row knobs: temperature T on both distributions ("Speculative decoding
// -- Hinglish notes", section "Temperature and Sampling"), or greedy
// verification (a draft is kept when it is the target's arg-max: "Inference:
// Sampling, the KV Cache, Speculative Decoding and int8", section
// "Speculative decoding"), for which only the target rows are read.
#include <cuda_runtime.h>

#include <climits>
#include <stdlib.h>
#include <mutex>
#include <type_traits>

#include "launch.h"
#include "row_ops.cuh"
#include "smp.h"

namespace smp {

#include "select.cuh"

// Statistics of one logit row, written by verify_pos_kernel.
struct PosStat {
  float m;          // row maximum
  int32_t flags;    // kRowNonFinite / kRowBadDraft / kRowBadParams
  uint64_t z;       // sum of fixed-point masses (filtered rows: Z_S); greedy rows: the arg-max id
  double ex;        // exp((z_x - m) / T) of the draft token (0 if none, or not kept)
  uint32_t kkey;    // kept set: order key > kkey, or == kkey with id <= kid
  uint32_t kid;     // (unfiltered rows: 0 and 0xFFFFFFFF, every token)
};

struct VerifyArgs {
  const void* p;
  const void* q;
  const int32_t* drafts;
  int batch;
  int k;
  int vocab;
  uint64_t seed;
  uint64_t offset;
  int32_t* accepted;
  int32_t* ids;
  int32_t* status;
  PosStat* ws;
  const smp_row_params* params;   // [batch] or nullptr (T = 1 on every row)
  float* alpha;                   // [batch, k] acceptance rates, or nullptr
  uint64_t row_base;              // global index of batch row 0 (Philox counter row)
  int exact_accept;               // decide every accept test on exact Z (tests of that path)
};

// How batch row b is verified: temperature T > 0 with or without filters,
// greedy, or an error row.  The knob rules are the sampler's: greedy (the
// flag, or T == 0) ignores the other knobs; otherwise the knobs must be valid
// sampling knobs, and the filters that are on apply to every p and q row.
struct RowMode {
  float temperature;
  bool greedy;
  bool bad;
  bool filtered;
};

template <bool kParams>
__device__ __forceinline__ RowMode row_mode(const VerifyArgs& a, int b) {
  RowMode md{1.0f, false, false, false};
  if (!kParams || a.params == nullptr) return md;
  const smp_row_params p = a.params[b];
  if (row_is_greedy(p)) {
    md.greedy = true;
    return md;
  }
  md.temperature = p.temperature;
  md.bad = !sampling_params_valid(p);
  md.filtered = (p.top_k > 0 && p.top_k < a.vocab) || p.top_p < 1.0f || (p.min_p > 0.0f && p.min_p < 1.0f);
  return md;
}

template <typename T>
__device__ __forceinline__ const T* logit_row(const VerifyArgs& a, int b, int j) {
  const size_t V = size_t(a.vocab);
  if (j <= a.k) return reinterpret_cast<const T*>(a.p) + (size_t(b) * (a.k + 1) + j) * V;
  return reinterpret_cast<const T*>(a.q) + (size_t(b) * a.k + (j - a.k - 1)) * V;
}

constexpr int kPosUnroll = 16;   // 16-byte loads in flight per thread in verify_pos_kernel
// ex2.approx.ftz.f32: largest relative error 1.46e-7, measured on GB300 over
// every binary32 input in [-126, 1] whose result is normal; with a margin:
constexpr double kEx2Err = 1.7e-7;
constexpr double kArgErr = 0.6931471805599453 * 0x1p-23;   // per unit |y|: y = (z - m) c rounded twice
constexpr uintptr_t kPosPrefetchChunk = 32768;        // one L2 prefetch request
constexpr uintptr_t kPosPrefetchBytes = 256 * 1024;   // most of a row prefetched before the wait

__device__ __forceinline__ uint4 load_stream(const uint4* p) {
  uint4 x;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w)
               : "l"(p));
  return x;
}

// Greedy verification's statistic of one target row: the maximum and its
// lowest id.  Each thread keeps (best, id) over its elements; its middle
// vectors come in increasing id order, so a vector replaces the best only
// when its maximum is strictly larger, and is then searched for the first
// element equal to it.  NaN never compares larger or equal, so it counts as
// -inf.  Returns the CTA's (maximum, lowest id holding it) in thread 0.
template <typename T>
__device__ __forceinline__ void greedy_row_argmax(const T* row, int Vn, int head, int tail0, const uint4* vec,
                                                  int nvec, float* redf, uint64_t* red64, float* m_out,
                                                  int* id_out) {
  using V = VecOps<T>;
  constexpr int kPer = V::kPer;
  const int tid = threadIdx.x;
  const uint32_t ninf = V::neg_inf();
  float best = -INFINITY;
  int bid = INT_MAX;
  auto consider = [&](float z, int i) {
    if (z > best || (z == best && i < bid)) {
      best = z;
      bid = i;
    }
  };
  for (int i = tid; i < head; i += kThreads) consider(Elem<T>::widen(row[i]), i);
  for (int v0 = 0; v0 < nvec; v0 += kThreads * kPosUnroll) {
    uint4 x[kPosUnroll];
#pragma unroll
    for (int u = 0; u < kPosUnroll; ++u) {
      const int i = v0 + tid + u * kThreads;
      x[u] = i < nvec ? load_stream(vec + i) : make_uint4(ninf, ninf, ninf, ninf);
    }
#pragma unroll
    for (int u = 0; u < kPosUnroll; ++u) {
      const float vm = V::finish(V::vmax(x[u]));
      if (vm > best) {
        const int base = head + (v0 + tid + u * kThreads) * kPer;
        int q0 = kPer - 1;
#pragma unroll
        for (int q = kPer - 1; q >= 0; --q)
          if (V::elem(x[u], q) == vm) q0 = q;
        best = vm;
        bid = base + q0;
      }
    }
  }
  for (int i = tail0 + tid; i < Vn; i += kThreads) consider(Elem<T>::widen(row[i]), i);
  const float m = block_max_f(best, redf);
  int cand = best == m ? bid : INT_MAX;
#pragma unroll
  for (int o = 16; o; o >>= 1) cand = min(cand, __shfl_xor_sync(0xFFFFFFFFu, cand, o));
  if ((tid & 31) == 0) red64[tid >> 5] = uint64_t(uint32_t(cand));
  cta_sync();
  if (tid == 0) {
    int id = INT_MAX;
    for (int w = 0; w < kWarps; ++w) id = min(id, int(uint32_t(red64[w])));
    *m_out = m;
    *id_out = id;
  }
}

// One CTA per logit row, one pass over it: the maximum and the fixed-point
// mass Z (online: a running maximum per thread, its sum rescaled when the
// maximum rises).  Thread 0 adds the draft token's mass (double-float
// exponential) and the flags.
// The statistic of one logit row of a filtered batch row: the row maximum,
// the kept set S of eq. 39.2 under the row's knobs (the sampler's exact
// selection over global memory), Z_S and the draft token's mass if it is in S.
constexpr int kVerifyTopU = 8;   // vectors in flight per thread in the light passes

template <typename T>
__device__ __forceinline__ void filtered_pos_stat(const VerifyArgs& a, const T* row, int pr, int b, int ipos,
                                                  const FloatPair* table) {
  __shared__ GenShared gs;   // histograms of the selection
  const int tid = threadIdx.x;
  const int Vn = a.vocab;
  const smp_row_params prm = a.params[b];
  // fmaxf skips NaN, which orders with -inf; -0 and +0 share a key
  float tmax = -INFINITY;
  gen_sweep<T, kVerifyTopU>(row, Vn, [&](int, float z) { tmax = fmaxf(tmax, z); });
  const uint32_t tkmax = order_key<T>(tmax);
  const uint32_t kmax = uint32_t(block_max_u64(uint64_t(tkmax), gs.red64));
  int flags = key_finite<T>(kmax) ? 0 : kRowNonFinite;
  int xd = -1;
  if (ipos < a.k) {
    xd = a.drafts[size_t(b) * a.k + ipos];
    if (xd < 0 || xd >= Vn) flags |= kRowBadDraft;
  }
  PosStat s;
  s.m = key_value<T>(kmax);
  s.z = 0;
  s.ex = 0.0;
  s.kkey = 0;
  s.kid = 0xFFFFFFFFu;
  if (!flags) {
    KeptSet ks;
    if (!topk_bounded(prm, Vn) || !gen_kept_set_topk<T, kVerifyTopU>(row, Vn, gs, table, prm, kmax, tkmax, &ks))
      ks = gen_kept_set<T>(row, Vn, gs, table, prm, kmax);
    s.z = ks.z_kept;
    s.kkey = ks.key;
    s.kid = ks.id_cut;
    if (ipos < a.k) s.ex = double(kept_mass<T>(ks, table, xd, Elem<T>::widen(row[xd]))) * (1.0 / double(kFixedOne));
  }
  s.flags = flags;
  if (tid == 0) a.ws[pr] = s;
}

// kParams: the call has per-row knobs (smp_spec_verify_params with params);
// without them the kernels carry neither the greedy nor the filtered code
// and no selection state in shared memory.
template <typename T, bool kParams>
__global__ void __launch_bounds__(kThreads, 2) verify_pos_kernel(VerifyArgs a) {
  using V = VecOps<T>;
  constexpr int kPer = V::kPer;
  __shared__ FloatPair table[64];
  __shared__ float redf[kWarps];
  __shared__ uint64_t red64[kWarps];
  const int tid = threadIdx.x;
  const int rows_per_b = 2 * a.k + 1;
  const int pr = int(blockIdx.x);
  const int b = pr / rows_per_b;
  const int j = pr % rows_per_b;
  const int Vn = a.vocab;
  // The row's aligned middle (up to kPosPrefetchBytes) is prefetched into L2
  // before the dependency wait: a prefetch changes no memory and L2 is the
  // point of coherence, so the previous kernel's writes still reach the loads
  // below; in a chain of calls it overlaps the previous call's resolve
  // kernel, which leaves HBM idle.
  if (tid == 0) {
    const T* prow = logit_row<T>(a, b, j);
    const uintptr_t p0 = (reinterpret_cast<uintptr_t>(prow) + 15) & ~uintptr_t(15);
    const uintptr_t p1 = (reinterpret_cast<uintptr_t>(prow) + size_t(Vn) * sizeof(T)) & ~uintptr_t(15);
    for (uintptr_t src = p0; src < p1 && src < p0 + kPosPrefetchBytes; src += kPosPrefetchChunk) {
      const uint32_t bytes = uint32_t(min(uintptr_t(kPosPrefetchChunk), p1 - src));
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
    }
  }
  grid_dependency_wait();
  allow_dependent_launch();
  // The status word is cleared here: only the resolve kernel, which waits
  // for this kernel to finish, ORs flags into it.
  if (blockIdx.x == 0 && tid == 0 && a.status) *a.status = 0;
  const RowMode md = row_mode<kParams>(a, b);
  if (md.bad || (md.greedy && j > a.k)) {
    // An error row's statistics carry the flag; greedy rows read no q row.
    if (tid == 0) {
      PosStat s;
      s.m = 0.0f;
      s.flags = md.bad ? kRowBadParams : 0;
      s.z = 0;
      s.ex = 0.0;
      s.kkey = 0;
      s.kid = 0xFFFFFFFFu;
      a.ws[pr] = s;
    }
    return;
  }
  if (tid < 64) table[tid] = kExp2Table[tid];

  const T* row = logit_row<T>(a, b, j);
  const int ipos = j <= a.k ? j : j - a.k - 1;   // draft position of this row
  if constexpr (kParams) {
    if (md.filtered) {
      cta_sync();   // the table is complete
      filtered_pos_stat<T>(a, row, pr, b, ipos, table);
      return;
    }
  }
  // The 16-byte aligned middle of the row, and the elements before and after it.
  const uintptr_t r0 = reinterpret_cast<uintptr_t>(row);
  const uintptr_t r1 = r0 + size_t(Vn) * sizeof(T);
  const uintptr_t m0 = (r0 + 15) & ~uintptr_t(15);
  const uintptr_t m1 = r1 & ~uintptr_t(15);
  const bool middle = m1 > m0;
  const int head = middle ? int((m0 - r0) / sizeof(T)) : Vn;
  const int tail0 = middle ? int((m1 - r0) / sizeof(T)) : Vn;
  const int nvec = middle ? int((m1 - m0) / 16) : 0;
  const uint4* vec = reinterpret_cast<const uint4*>(m0);
  const uint32_t ninf = V::neg_inf();

  // The draft token's logit, requested now so that the load overlaps the stream.
  int xd = -1;
  float zx = -INFINITY;
  if (tid == 0 && ipos < a.k) {
    xd = a.drafts[size_t(b) * a.k + ipos];
    if (xd >= 0 && xd < Vn && !md.greedy) zx = Elem<T>::widen(row[xd]);
  }

  if (md.greedy) {   // a target row of a greedy row: its arg-max, and the draft's range
    float gm;
    int gid;
    greedy_row_argmax<T>(row, Vn, head, tail0, vec, nvec, redf, red64, &gm, &gid);
    if (tid == 0) {
      PosStat s;
      s.m = gm;
      s.flags = (isfinite(gm) ? 0 : kRowNonFinite) | (ipos < a.k && (xd < 0 || xd >= Vn) ? kRowBadDraft : 0);
      s.z = uint64_t(uint32_t(gid));
      s.ex = 0.0;
      s.kkey = 0;
      s.kid = 0xFFFFFFFFu;
      a.ws[pr] = s;
    }
    return;
  }

  // One pass over the row: each thread keeps a running maximum (rs.m) and
  // the binary32 sum st of exp(z - rs.m) over its elements, rescaled when the
  // maximum of a group of kPosUnroll vectors raises it.  The exponentials of
  // a group are summed as trees (per vector, then over the group).
  RowScale rs = make_row_scale(-INFINITY, md.temperature);
  float st = 0.0f;
  auto raise_to = [&](float g) {   // g > rs.m
    st = rs.m > -INFINITY ? __fmul_rn(st, exp_fast(rs.m, RowScale{g, rs.c_hi, rs.c_lo})) : 0.0f;
    rs.m = g;
  };
  for (int v0 = 0; v0 < nvec; v0 += kThreads * kPosUnroll) {
    uint4 x[kPosUnroll];
#pragma unroll
    for (int u = 0; u < kPosUnroll; ++u) {
      const int i = v0 + tid + u * kThreads;
      x[u] = i < nvec ? load_stream(vec + i) : make_uint4(ninf, ninf, ninf, ninf);
    }
    uint32_t pm = ninf;
#pragma unroll
    for (int u = 0; u < kPosUnroll; ++u) pm = V::max2(pm, V::vmax(x[u]));
    const float gm = V::finish(pm);
    if (gm > rs.m) raise_to(gm);
    if (rs.m > -INFINITY) {
      float vs[kPosUnroll];
#pragma unroll
      for (int u = 0; u < kPosUnroll; ++u) {
        float e[kPer];
#pragma unroll
        for (int q = 0; q < kPer; ++q) e[q] = exp_fast(V::elem(x[u], q), rs);
#pragma unroll
        for (int w = kPer / 2; w > 0; w /= 2)
#pragma unroll
          for (int q = 0; q < w; ++q) e[q] += e[q + w];
        vs[u] = e[0];
      }
#pragma unroll
      for (int w = kPosUnroll / 2; w > 0; w /= 2)
#pragma unroll
        for (int u = 0; u < w; ++u) vs[u] += vs[u + w];
      st += vs[0];
    }
  }
  auto edge = [&](float z) {
    if (z > rs.m) raise_to(z);
    if (rs.m > -INFINITY) st += exp_fast(z, rs);
  };
  for (int i = tid; i < head; i += kThreads) edge(Elem<T>::widen(row[i]));
  for (int i = tail0 + tid; i < Vn; i += kThreads) edge(Elem<T>::widen(row[i]));
  const float m = block_max_f(rs.m, redf);
  int flags = 0;
  if (!isfinite(m)) flags |= kRowNonFinite;
  const RowScale rm = make_row_scale(m, md.temperature);

  // Z = sum over threads of st * exp(rs.m - m): each thread's share in
  // fixed point once, summed exactly.  Relative error about 3e-7.
  float zf = 0.0f;
  if (!flags && rs.m > -INFINITY) zf = __fmul_rn(st, exp_fast(rs.m, rm));
  uint64_t z = __float2ull_rn(__fmul_rn(zf, float(kFixedOne)));
  z = warp_sum<uint64_t>(z);
  if ((tid & 31) == 0) red64[tid >> 5] = z;
  cta_sync();
  if (tid == 0) {
    uint64_t tot = 0;
    for (int w = 0; w < kWarps; ++w) tot += red64[w];
    double ex = 0.0;
    if (ipos < a.k) {
      if (xd < 0 || xd >= Vn) flags |= kRowBadDraft;
      else if (!flags) ex = mass_double(zx, rm, table);
    }
    PosStat st;
    st.m = m;
    st.flags = flags;
    st.z = tot;
    st.ex = ex;
    st.kkey = 0;
    st.kid = 0xFFFFFFFFu;
    a.ws[pr] = st;
  }
}

constexpr int kResolveThreads = 256;
constexpr int kResolveWarps = kResolveThreads / 32;
constexpr int kResolveMaxCluster = 8;   // CTAs (one cluster) per batch row

// Exclusive prefix over the CTA of one u64 per thread (thread order), and the total.
__device__ __forceinline__ uint64_t resolve_scan(uint64_t v, uint64_t* warp_tot, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t incl = warp_inclusive_scan<uint64_t>(v);
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  uint64_t before = incl - v, all = 0;
  for (int w = 0; w < kResolveWarps; ++w) {
    const uint64_t t = warp_tot[w];
    if (w < warp) before += t;
    all += t;
  }
  __syncthreads();   // warp_tot may be written again
  *total = all;
  return before;
}

// Sum of one u64 per CTA of the cluster (v, the same in every thread of the
// CTA): this CTA's exclusive prefix (cluster rank order) and the cluster
// total.  Lane r of warp 0 stores v into slots[rank] of the CTA of rank r; one
// cluster barrier (release / acquire) makes every value local, and no CTA
// touches a peer's memory after it.  Every CTA of the cluster must have
// passed a cluster barrier before the first call (peers have started), and
// each call needs its own `slots` array of kResolveMaxCluster words.
__device__ __forceinline__ uint64_t cluster_prefix(uint64_t v, uint64_t* slots, uint64_t* bc, uint64_t* total) {
  const uint32_t rank = cluster_rank(), n = cluster_size();
  if (threadIdx.x < n) st_cluster_u64(map_rank(smem_addr(slots + rank), threadIdx.x), v);
  hw_cluster_sync();
  if (threadIdx.x < 32) {
    const uint32_t r = threadIdx.x;
    const uint64_t t = r < n ? slots[r] : 0ull;
    const uint64_t before = warp_sum<uint64_t>(r < rank ? t : 0ull);
    const uint64_t all = warp_sum<uint64_t>(t);
    if (r == 0) {
      bc[0] = before;
      bc[1] = all;
    }
  }
  __syncthreads();
  *total = bc[1];
  return bc[0];
}

// Per-position state of the acceptance rates alpha_i = sum_x min(p_i, q_i)
// (shared memory of the resolve kernel's knob instance, only when asked for).
struct AlphaShared {
  float m[2][SMP_MAX_DRAFT];            // maxima of p_i and q_i
  float inv_z[2][SMP_MAX_DRAFT];        // 2^F / Z of p_i and q_i (binary32)
  uint32_t kept[4][SMP_MAX_DRAFT];      // kept sets of p_i and q_i: (key, id) each
  unsigned long long cta[SMP_MAX_DRAFT];                       // this CTA's sums
  unsigned long long slots[kResolveMaxCluster][SMP_MAX_DRAFT];  // rank 0: every CTA's sums
};

__device__ __forceinline__ AlphaShared& alpha_shared() {
  __shared__ AlphaShared s;
  return s;
}

// rn(r * 2^52) for 0 <= r <= 1 from two 32-bit conversions: s = r * 2^28 <= 2^28
// splits exactly into its integer part and fraction; the fraction times 2^24
// rounds like the whole (the integer part times 2^24 is even).
__device__ __forceinline__ uint64_t fixed52(float r) {
  const float sc = __fmul_rn(r, 0x1p28f);
  const float hi = truncf(sc);
  return (uint64_t(__float2uint_rz(hi)) << 24) + __float2uint_rn(__fmul_rn(__fsub_rn(sc, hi), 0x1p24f));
}

// One cluster per batch row: the accept tests of eq. 39.3 in position order,
// then the replacement draw from max(0, p_j - q_j) (eq. 39.4) at the first
// rejection j, or the bonus draw from p_K.  Thread g of the cluster (rank-major)
// owns the token ids [g C, (g + 1) C): weights are 52-bit fixed point with
// exact integer sums; CTA and cluster scans find the chunk that holds the
// draw, and warp 0 of its CTA walks it.
template <typename T, bool kParams>
__global__ void __launch_bounds__(kResolveThreads, 2) verify_resolve_kernel(VerifyArgs a) {
  __shared__ int32_t decision[3];   // first rejection j, row flags, an undecided test
  __shared__ uint64_t ez_zp[SMP_MAX_DRAFT], ez_zq[SMP_MAX_DRAFT];   // exact Z of retested positions
  __shared__ int ez_have[SMP_MAX_DRAFT];
  __shared__ uint64_t ez_wq[kResolveWarps];
  __shared__ uint64_t ez_slots[2][kResolveMaxCluster];
  __shared__ FloatPair table[64];   // 2^(j/64) for the exact retest's exponentials
  __shared__ float inv_z[2];        // 2^F / Z of the drawn row's p and q (binary32)
  __shared__ float row_m[2];        // the drawn row's p and q maxima
  __shared__ uint32_t kept_desc[4]; // the drawn row's p and q kept sets (key, id) when filtered
  __shared__ uint64_t warp_tot[kResolveWarps];
  __shared__ uint64_t cta_slots[2][kResolveMaxCluster];   // one array per cluster_prefix call
  __shared__ uint64_t cta_bc[2];
  __shared__ int owner;             // thread whose ids hold the draw
  __shared__ uint64_t owner_before;
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank(), nranks = cluster_size();
  const int b = int(blockIdx.x / nranks);
  const int K = a.k;
  const int V = a.vocab;
  const int rows_per_b = 2 * K + 1;
  const PosStat* st = a.ws + size_t(b) * rows_per_b;
  // The uniforms depend on nothing the position kernel writes: drawn while it runs.
  const uint64_t grow = a.row_base + uint64_t(b);
  const uint64_t u_acc = threadIdx.x < K ? uniform53(a.seed, a.offset, grow, uint64_t(threadIdx.x)) : 0ull;
  const uint64_t u53 = uniform53(a.seed, a.offset, grow, uint64_t(K));
  hw_cluster_sync();        // every CTA of the cluster has started (remote stores below)
  grid_dependency_wait();   // the position statistics come from verify_pos_kernel
  allow_dependent_launch();
  const RowMode md = row_mode<kParams>(a, b);
  if (tid < 64) table[tid] = kExp2Table[tid];

  // Greedy verification (and error rows): lane i compares draft i with the
  // target's arg-max of position i; the first mismatch j emits the arg-max of
  // position j (position K when every draft matches).  Rank 0's warp 0 writes
  // the row; no uniform and no other CTA is needed.
  if (md.greedy || md.bad) {
    if (rank == 0 && tid < 32) {
      const int i = tid;
      PosStat P{};
      if (i <= K) P = st[i];
      int fl = (i <= K ? P.flags : 0) | (md.bad ? kRowBadParams : 0);
      for (int o = 16; o; o >>= 1) fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, o);
      const int top = int(uint32_t(P.z));
      const int draft = i < K ? a.drafts[size_t(b) * K + i] : -1;
      const uint32_t miss = __ballot_sync(0xFFFFFFFFu, i < K && draft != top);
      const int jr = miss ? __ffs(miss) - 1 : K;
      const int top_j = __shfl_sync(0xFFFFFFFFu, top, jr);
      if (i <= K) a.ids[size_t(b) * (K + 1) + i] = fl ? -1 : i < jr ? draft : i == jr ? top_j : -1;
      if (a.alpha && i < K) a.alpha[size_t(b) * K + i] = __int_as_float(0x7FC00000);   // no q compared
      if (i == 0) {
        a.accepted[b] = fl ? -1 : jr;
        if (fl && a.status) atomicOr(a.status, fl & (kRowNonFinite | kRowBadDraft | kRowBadParams));
      }
    }
    return;
  }

  // Thread g of the cluster owns ids [c0, c1): a whole number of 16-byte
  // groups of the row (rows whose base is not 16-byte aligned fall back to
  // element loads).
  constexpr int kPer = 16 / int(sizeof(T));
  const int nthreads = int(nranks) * kResolveThreads;
  const int per = (V + nthreads - 1) / nthreads;
  const int chunk = (per + kPer - 1) / kPer * kPer;
  const int g = int(rank) * kResolveThreads + tid;
  const int c0 = min(V, g * chunk), c1 = min(V, c0 + chunk);

  // Worst-case relative error of the position kernel's Z (unfiltered rows):
  // every exponential is ex2.approx (largest relative error 1.46e-7, measured
  // over every binary32 input in [-126, 1] on GB300; kEx2Err with a margin),
  // applied once per element, once per rescaling of a thread's running sum
  // (at most one per group of kPosUnroll vectors, plus one for the row's
  // edges) and once to scale the thread's sum to the row maximum; the
  // rounding of each argument y = (z - m) log2(e) / T, relative to y, whose
  // mean |y| under the row's distribution is at most log2(V) (it equals the
  // entropy H(p) minus log2 Z, Z >= 1), twice for the shifts to new maxima;
  // the binary32 sums (a tree over a group, then one addition per group and
  // one product per rescaling).
  const int groups = (V * int(sizeof(T)) / 16 + kThreads * kPosUnroll - 1) / (kThreads * kPosUnroll) + 1;
  const float z_err = md.filtered ? 0.0f
                                  : float(groups + 2) * float(kEx2Err) + 2.0f * float(kArgErr) * log2f(float(V)) +
                                        float(2 * groups + 9) * 0x1p-24f + 1e-10f;

  // Accept tests u_i < p_i(x) / max(q_i(x), 1e-300), one lane per position
  // (K <= 32), as the product form u_i * max(q, 1e-300) < p with
  // p = ex_p / (Z_p 2^-F), q = ex_q / (Z_q 2^-F); the first failing position
  // is the rejection.  A test whose two sides are closer than the error of
  // the fast Z allows is decided again on Z recomputed exactly (double-float
  // exponentials summed as integers over the cluster).  Every CTA of the
  // cluster decides alike.
  PosStat P{}, Q{};
  if (tid < 32) {
    if (tid <= K) P = st[tid];
    if (tid < K) Q = st[K + 1 + tid];
    if (tid < K) ez_have[tid] = 0;
  }
  for (int iter = 0; iter <= K; ++iter) {
    if (tid < 32) {
      const int i = tid;
      int fl = (i <= K ? P.flags : 0) | (i < K ? Q.flags : 0);
      for (int o = 16; o; o >>= 1) fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, o);
      bool reject = false, unsure = false;
      if (!fl && i < K) {
        const bool exact = ez_have[i] != 0;
        const double zp = double(exact ? ez_zp[i] : P.z) * (1.0 / double(kFixedOne));
        const double zq = double(exact ? ez_zq[i] : Q.z) * (1.0 / double(kFixedOne));
        const double u = double(u_acc) * 0x1p-53;
        // u * max(ex_q / zq, 1e-300) < ex_p / zp, multiplied through by zp * zq > 0
        const double lhs = Q.ex > 0.0 ? u * Q.ex * zp : u * 1e-300 * zp * zq;
        const double rhs = P.ex * zq;
        reject = !(lhs < rhs);
        unsure = !exact && (a.exact_accept || fabs(lhs - rhs) <= double(2.0f * z_err + 1e-12f) * fmax(lhs, rhs));
      }
      const uint32_t hit = __ballot_sync(0xFFFFFFFFu, reject || unsure);
      const int jr = hit ? __ffs(hit) - 1 : K;
      const bool jr_unsure = __shfl_sync(0xFFFFFFFFu, unsure ? 1 : 0, jr < 32 ? jr : 0) != 0;
      const bool undecided = !fl && jr < K && jr_unsure;
      if (tid == 0) {
        decision[0] = jr;
        decision[1] = fl;
        decision[2] = undecided ? 1 : 0;
      }
      if (!undecided) {
        // For the drawn row, the maxima and reciprocals of Z the draw needs,
        // once, in binary32 (within an ulp of 2^F / Z; FP64 is slow on this
        // part); the acceptance rates' per-position state.
        if (i == jr && !fl) {
          row_m[0] = P.m;
          inv_z[0] = __fdiv_rn(float(kFixedOne), __ull2float_rn(P.z));
          row_m[1] = jr < K ? Q.m : P.m;
          inv_z[1] = jr < K ? __fdiv_rn(float(kFixedOne), __ull2float_rn(Q.z)) : inv_z[0];
          kept_desc[0] = P.kkey;
          kept_desc[1] = P.kid;
          kept_desc[2] = jr < K ? Q.kkey : P.kkey;
          kept_desc[3] = jr < K ? Q.kid : P.kid;
        }
        if constexpr (kParams) {
          if (a.alpha && i < K && !fl) {
            AlphaShared& as = alpha_shared();
            as.m[0][i] = P.m;
            as.m[1][i] = Q.m;
            as.inv_z[0][i] = __fdiv_rn(float(kFixedOne), __ull2float_rn(P.z));
            as.inv_z[1][i] = __fdiv_rn(float(kFixedOne), __ull2float_rn(Q.z));
            as.kept[0][i] = P.kkey;
            as.kept[1][i] = P.kid;
            as.kept[2][i] = Q.kkey;
            as.kept[3][i] = Q.kid;
            as.cta[i] = 0;
          }
        }
      }
    }
    __syncthreads();
    if (!decision[2]) break;
    // Exact Z of the undecided position's p and q rows.
    const int pos = decision[0];
    const RowScale sp = make_row_scale(st[pos].m, md.temperature);
    const RowScale sq = make_row_scale(st[K + 1 + pos].m, md.temperature);
    const T* pr = logit_row<T>(a, b, pos);
    const T* qr = logit_row<T>(a, b, K + 1 + pos);
    uint64_t ep = 0, eq = 0;
    for (int i = c0; i < c1; ++i) {
      ep += mass_fixed(Elem<T>::widen(pr[i]), sp, table);
      eq += mass_fixed(Elem<T>::widen(qr[i]), sq, table);
    }
    uint64_t tp = 0, tq = 0, cta_p = 0, cta_q = 0;
    ep = warp_sum<uint64_t>(ep);
    eq = warp_sum<uint64_t>(eq);
    if ((tid & 31) == 0) {
      warp_tot[tid >> 5] = ep;
      ez_wq[tid >> 5] = eq;
    }
    __syncthreads();
    for (int w = 0; w < kResolveWarps; ++w) {
      cta_p += warp_tot[w];
      cta_q += ez_wq[w];
    }
    __syncthreads();
    cluster_prefix(cta_p, ez_slots[0], cta_bc, &tp);
    cluster_prefix(cta_q, ez_slots[1], cta_bc, &tq);
    if (tid == 0) {
      ez_zp[pos] = tp;
      ez_zq[pos] = tq;
      ez_have[pos] = 1;
    }
    __syncthreads();
  }
  __syncthreads();
  const int jrej = decision[0];
  const int flags = decision[1];
  if (flags) {
    if (rank == 0 && tid == 0) {
      a.accepted[b] = -1;
      for (int i = 0; i <= K; ++i) a.ids[size_t(b) * (K + 1) + i] = -1;
      if (a.alpha)
        for (int i = 0; i < K; ++i) a.alpha[size_t(b) * K + i] = __int_as_float(0x7FC00000);
      if (a.status) atomicOr(a.status, flags & (kRowNonFinite | kRowBadDraft | kRowTimeout | kRowBadParams));
    }
    return;
  }

  const bool residual = jrej < K;
  const T* prow = logit_row<T>(a, b, jrej);               // p_j (or p_K for the bonus)
  const T* qrow = residual ? logit_row<T>(a, b, K + 1 + jrej) : prow;
  const RowScale rp = make_row_scale(row_m[0], md.temperature);
  const RowScale rq = make_row_scale(row_m[1], md.temperature);
  // Weights in fixed point with 52 fraction bits: max(0, p - q) with
  // p = e_p / Z_p and q = e_q / Z_q in binary32 (eq. 39.4), or e_p / Z_p for a
  // draw from p.  r * 2^52 is the binary32 r exactly for r >= 2^-28 (below,
  // within 2^-53), and the row's total stays below 2^53 because the p sum to
  // 1.  The sums are exact integers, so the scans and the walk agree.
  bool use_p = !residual;
  const float inv_zp = inv_z[0];
  const float inv_zq = inv_z[1];
  // Filtered rows: p~ and q~ are 0 outside their kept sets (eq. 39.2).
  const bool filt = md.filtered;
  KeptSet kp, kq;
  kp.key = kept_desc[0];
  kp.id_cut = kept_desc[1];
  kq.key = kept_desc[2];
  kq.id_cut = kept_desc[3];
  // kFilt (a std::bool_constant) selects the membership test at compile
  // time, so unfiltered rows run the loops without it.
  auto weight_of = [&](auto kFilt, int id, float zp, float zq) -> uint64_t {
    float p = __fmul_rn(exp_fast(zp, rp), inv_zp);
    float q = use_p ? 0.0f : __fmul_rn(exp_fast(zq, rq), inv_zq);
    if constexpr (decltype(kFilt)::value) {
      if (!in_kept_set(kp, order_key<T>(zp), uint32_t(id))) p = 0.0f;
      if (!in_kept_set(kq, order_key<T>(zq), uint32_t(id))) q = 0.0f;
    }
    const float r = use_p ? p : fmaxf(0.0f, __fsub_rn(p, q));
    return fixed52(r);
  };
  constexpr int kGroups = 16 / kPer;   // groups of kPer ids in flight per thread (16 ids)
  // Sum of w(id, z_p, z_q) over the thread's ids of one row pair (q not read
  // when read_q is false): all its vectors requested first, then a rolled
  // loop over the groups (this code runs once per CTA, cold in the
  // instruction cache, so it is kept short).
  // w returns a 52-bit fixed-point weight, summed as is, or a binary32 value,
  // summed in binary32 over each group of 16 ids and then converted once.
  auto pair_sum = [&](const T* pr_, const T* qr_, bool read_q, auto&& w) -> uint64_t {
    using Acc = decltype(w(0, 0.0f, 0.0f));
    const bool vok = ((reinterpret_cast<uintptr_t>(pr_) | reinterpret_cast<uintptr_t>(qr_)) & 15) == 0;
    uint64_t sum = 0;
    const uint32_t ninf = VecOps<T>::neg_inf();
    for (int g0 = c0; g0 < c1; g0 += kGroups * kPer) {
      uint4 xp[kGroups], xq[kGroups];
#pragma unroll
      for (int gi = 0; gi < kGroups; ++gi) {
        const int gg = g0 + gi * kPer;
        xp[gi] = make_uint4(ninf, ninf, ninf, ninf);
        xq[gi] = xp[gi];
        if (gg < c1 && vok && gg + kPer <= V) {
          xp[gi] = __ldg(reinterpret_cast<const uint4*>(pr_ + gg));
          xq[gi] = read_q ? __ldg(reinterpret_cast<const uint4*>(qr_ + gg)) : xp[gi];
        }
      }
      Acc gsum = 0;
#pragma unroll 1
      for (int gi = 0; gi < kGroups; ++gi) {
        const int gg = g0 + gi * kPer;
        if (gg >= c1) break;
        uint4 vp = xp[0], vq = xq[0];
#pragma unroll
        for (int k2 = 1; k2 < kGroups; ++k2)
          if (gi == k2) {
            vp = xp[k2];
            vq = xq[k2];
          }
        const bool full = vok && gg + kPer <= V;
#pragma unroll
        for (int e = 0; e < kPer; ++e) {
          float zp = VecOps<T>::elem(vp, e), zq = VecOps<T>::elem(vq, e);
          if (!full) {   // a row not 16-byte aligned, or its last ids
            zp = gg + e < c1 ? Elem<T>::widen(pr_[gg + e]) : -INFINITY;
            zq = gg + e < c1 ? Elem<T>::widen(qr_[gg + e]) : -INFINITY;
          }
          gsum += w(gg + e, zp, zq);
        }
      }
      if constexpr (std::is_same<Acc, float>::value) sum += fixed52(gsum);
      else sum += gsum;
    }
    return sum;
  };
  auto chunk_sum = [&](auto kFilt) -> uint64_t {
    return pair_sum(prow, qrow, !use_p, [&](int id, float zp, float zq) { return weight_of(kFilt, id, zp, zq); });
  };
  auto chunk_sum_row = [&]() { return filt ? chunk_sum(std::true_type{}) : chunk_sum(std::false_type{}); };
  uint64_t local = chunk_sum_row(), cta_total = 0, total = 0;
  uint64_t before = resolve_scan(local, warp_tot, &cta_total);
  uint64_t cta_before = cluster_prefix(cta_total, cta_slots[0], cta_bc, &total);
  if (residual && total == 0) {   // zero residual mass (rounding only): draw from p_j
    use_p = true;
    local = chunk_sum_row();
    before = resolve_scan(local, warp_tot, &cta_total);
    cta_before = cluster_prefix(cta_total, cta_slots[1], cta_bc, &total);
  }
  before += cta_before;
  const uint64_t t = uint64_t((u128(u53) * total) >> 53);
  // The chunk whose cumulative interval holds t is walked by warp 0 of its
  // CTA, 32 ids per step: weights, a warp scan, the first id whose running
  // total passes t.
  if (tid == 0) owner = -1;
  __syncthreads();
  if (local > 0 && t >= before && t - before < local) {
    owner = tid;
    owner_before = before;
  }
  __syncthreads();
  if (owner >= 0 && tid < 32) {
    const int lane = tid;
    const int o0 = min(V, (int(rank) * kResolveThreads + owner) * chunk), o1 = min(V, o0 + chunk);
    uint64_t run = owner_before;
    for (int base = o0; base < o1; base += 32) {
      const int i = base + lane;
      const float zp = i < o1 ? Elem<T>::widen(prow[i]) : 0.0f, zq = i < o1 ? Elem<T>::widen(qrow[i]) : 0.0f;
      const uint64_t w = i >= o1 ? 0ull
                         : filt  ? weight_of(std::true_type{}, i, zp, zq)
                                 : weight_of(std::false_type{}, i, zp, zq);
      const uint64_t incl = warp_inclusive_scan<uint64_t>(w);
      const uint32_t hit = __ballot_sync(0xFFFFFFFFu, i < o1 && run + incl > t);
      if (hit) {
        if (lane == __ffs(hit) - 1) a.ids[size_t(b) * (K + 1) + jrej] = i;
        break;
      }
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  if (rank == 0 && tid == 0) {
    a.accepted[b] = jrej;
    for (int i = 0; i < jrej; ++i) a.ids[size_t(b) * (K + 1) + i] = a.drafts[size_t(b) * K + i];
    for (int i = jrej + 1; i <= K; ++i) a.ids[size_t(b) * (K + 1) + i] = -1;
  }

  // Acceptance rates alpha_i = sum_x min(p_i(x), q_i(x)) for every draft
  // position ("Decoding & Speculative Sampling", section 39.4, Listing 39.5),
  // on the compared distributions (binary32 p and q; binary32 sums over
  // groups of 16 ids, within 16 units of 2^-24 of each group's sum, then
  // 52-bit fixed-point sums over the same id chunks as the draw).  The p_i
  // and q_i rows were read by the position kernel just before and are
  // normally served by L2.
  if constexpr (kParams) {
    if (a.alpha) {
      AlphaShared& as = alpha_shared();
      for (int i = 0; i < K; ++i) {
        const RowScale sp = make_row_scale(as.m[0][i], md.temperature);
        const RowScale sq = make_row_scale(as.m[1][i], md.temperature);
        const float izp = as.inv_z[0][i], izq = as.inv_z[1][i];
        KeptSet kpi, kqi;
        kpi.key = as.kept[0][i];
        kpi.id_cut = as.kept[1][i];
        kqi.key = as.kept[2][i];
        kqi.id_cut = as.kept[3][i];
        uint64_t sum = pair_sum(logit_row<T>(a, b, i), logit_row<T>(a, b, K + 1 + i), true,
                                [&](int id, float zp, float zq) -> float {
                                  float p = __fmul_rn(exp_fast(zp, sp), izp);
                                  float q = __fmul_rn(exp_fast(zq, sq), izq);
                                  if (filt) {
                                    if (!in_kept_set(kpi, order_key<T>(zp), uint32_t(id))) p = 0.0f;
                                    if (!in_kept_set(kqi, order_key<T>(zq), uint32_t(id))) q = 0.0f;
                                  }
                                  return fminf(p, q);
                                });
        sum = warp_sum<uint64_t>(sum);
        if ((tid & 31) == 0 && sum) atomicAdd(&as.cta[i], (unsigned long long)sum);
      }
      __syncthreads();
      if (tid < K) st_cluster_u64(map_rank(smem_addr(&as.slots[rank][tid]), 0), as.cta[tid]);
      hw_cluster_sync();   // every CTA's sums are in rank 0's slots
      if (rank == 0 && tid < K) {
        uint64_t tot = 0;
        for (uint32_t r = 0; r < nranks; ++r) tot += as.slots[r][tid];
        a.alpha[size_t(b) * K + tid] = float(double(tot) * 0x1p-52);
      }
    }
  }
}

// ------------------------------------------------------------------ host side

template <typename T>
static smp_status launch_verify(VerifyArgs a, cudaStream_t stream) {
  const int dev = current_device();
  if (dev < 0) return fail_cuda(cudaGetLastError());
  const int rows = a.batch * (2 * a.k + 1);
  LaunchShape ls;   // one CTA per logit row, then one per batch row; no dynamic shared memory
  ls.pdl = true;
  cudaError_t err;
  const bool knobs = a.params != nullptr || a.alpha != nullptr;   // the instances with per-row knobs
  const void* pos = knobs ? reinterpret_cast<const void*>(&verify_pos_kernel<T, true>)
                          : reinterpret_cast<const void*>(&verify_pos_kernel<T, false>);
  const void* resolve = knobs ? reinterpret_cast<const void*>(&verify_resolve_kernel<T, true>)
                              : reinterpret_cast<const void*>(&verify_resolve_kernel<T, false>);
  err = launch_cluster(pos, dim3(rows), dim3(kThreads), ls,
                       stream, &a);
  if (err != cudaSuccess) return fail_cuda(err);
  // Enough CTAs per batch row to cover the GPU twice over, at most one portable cluster.
  LaunchShape lr = ls;
  const int sms = device_sms(dev);
  while (lr.cluster < kResolveMaxCluster && int64_t(a.batch) * lr.cluster < 2 * sms) lr.cluster *= 2;
  if (forced_cluster() && forced_cluster() <= kResolveMaxCluster) lr.cluster = forced_cluster();
  err = launch_cluster(resolve, dim3(a.batch * lr.cluster),
                       dim3(kResolveThreads), lr, stream, &a);
  if (err != cudaSuccess) return fail_cuda(err);
  return SMP_OK;
}

}  // namespace smp

extern "C" size_t smp_spec_verify_workspace_bytes(int32_t batch, int32_t k) {
  if (batch <= 0 || batch > (1 << 20) || k < 1 || k > SMP_MAX_DRAFT) return 0;
  return size_t(batch) * size_t(2 * k + 1) * sizeof(smp::PosStat);
}

namespace smp {

// Every verifier entry point: argument checks, then the two kernels.
static smp_status verify_entry(const void* p_logits, const void* q_logits, const int32_t* draft_ids, int32_t batch,
                               int32_t k, int32_t vocab, smp_dtype dtype, const smp_row_params* params, uint64_t seed,
                               uint64_t offset, uint64_t row_base, int32_t* out_accepted_len, int32_t* out_ids,
                               float* out_alpha, int32_t* status, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (dtype != SMP_F32 && dtype != SMP_BF16) return SMP_ERR_DTYPE;
  if (!p_logits || !q_logits || !draft_ids || !out_accepted_len || !out_ids) return SMP_ERR_INVALID_ARG;
  if (batch <= 0 || batch > (1 << 20) || k < 1 || k > SMP_MAX_DRAFT || vocab <= 0)
    return SMP_ERR_INVALID_ARG;
  if (vocab > SMP_MAX_VOCAB) return SMP_ERR_UNSUPPORTED;
  const size_t elem = dtype == SMP_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(p_logits) % elem || reinterpret_cast<uintptr_t>(q_logits) % elem)
    return SMP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(draft_ids) % 4 || reinterpret_cast<uintptr_t>(out_ids) % 4 ||
      reinterpret_cast<uintptr_t>(out_accepted_len) % 4 || reinterpret_cast<uintptr_t>(params) % 4 ||
      reinterpret_cast<uintptr_t>(out_alpha) % 4 || reinterpret_cast<uintptr_t>(status) % 4)
    return SMP_ERR_INVALID_ARG;
  const size_t need = smp_spec_verify_workspace_bytes(batch, k);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 8)
    return SMP_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  VerifyArgs a{};
  a.p = p_logits;
  a.q = q_logits;
  a.drafts = draft_ids;
  a.batch = batch;
  a.k = k;
  a.vocab = vocab;
  a.seed = seed;
  a.offset = offset;
  a.row_base = row_base;
  a.exact_accept = getenv("SMP_VERIFY_EXACT_ACCEPT") != nullptr;
  a.accepted = out_accepted_len;
  a.ids = out_ids;
  a.status = status;
  a.ws = reinterpret_cast<PosStat*>(workspace);
  a.params = params;
  a.alpha = out_alpha;
  if (dtype == SMP_F32) return launch_verify<float>(a, st);
  return launch_verify<uint16_t>(a, st);
}

}  // namespace smp

extern "C" smp_status smp_spec_verify_params(const void* p_logits, const void* q_logits,
                                             const int32_t* draft_ids, int32_t batch, int32_t k,
                                             int32_t vocab, smp_dtype dtype, const smp_row_params* params,
                                             uint64_t seed, uint64_t offset, int32_t* out_accepted_len,
                                             int32_t* out_ids, float* out_alpha, int32_t* status,
                                             void* workspace, size_t workspace_bytes, void* stream) {
  return smp::verify_entry(p_logits, q_logits, draft_ids, batch, k, vocab, dtype, params, seed, offset, 0,
                           out_accepted_len, out_ids, out_alpha, status, workspace, workspace_bytes, stream);
}

extern "C" smp_status smp_spec_verify_rows(const void* p_logits, const void* q_logits, const int32_t* draft_ids,
                                           int32_t batch, int32_t k, int32_t vocab, smp_dtype dtype,
                                           const smp_row_params* params, uint64_t seed, uint64_t offset,
                                           uint64_t row_base, int32_t* out_accepted_len, int32_t* out_ids,
                                           float* out_alpha, int32_t* status, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  return smp::verify_entry(p_logits, q_logits, draft_ids, batch, k, vocab, dtype, params, seed, offset, row_base,
                           out_accepted_len, out_ids, out_alpha, status, workspace, workspace_bytes, stream);
}

extern "C" smp_status smp_spec_verify(const void* p_logits, const void* q_logits,
                                      const int32_t* draft_ids, int32_t batch, int32_t k, int32_t vocab,
                                      smp_dtype dtype, uint64_t seed, uint64_t offset,
                                      int32_t* out_accepted_len, int32_t* out_ids, int32_t* status,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  return smp_spec_verify_params(p_logits, q_logits, draft_ids, batch, k, vocab, dtype, nullptr, seed, offset,
                                out_accepted_len, out_ids, nullptr, status, workspace, workspace_bytes, stream);
}

// ------------------------------------------------------------------ allocation-free variant
//
// For callers that cannot allocate device memory when they verify (allocator
// or pool callbacks, runtimes that forbid cudaMalloc while serving, loops that
// must not let cudaMalloc / cudaFree synchronise the device), the workspace of
// smp_spec_verify can live in this fixed array instead.  Every GPU that loads
// the library holds it until the process exits.  All calls on a device share
// it: each call writes every entry before it reads it, and calls that overlap
// on the GPU race.

namespace smp {

constexpr size_t kStaticVerifyScratchBytes = SMP_STATIC_VERIFY_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_verify_scratch[kStaticVerifyScratchBytes];

// Device address of g_verify_scratch on `dev`, looked up once per device with
// that device current (in host code the array's name is not a device address).
static void* static_scratch_address(int dev, cudaError_t* err) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  *err = cudaSuccess;
  return addr[dev];
}

}  // namespace smp

extern "C" smp_status smp_spec_verify_static(const void* p_logits, const void* q_logits,
                                             const int32_t* draft_ids, int32_t batch, int32_t k,
                                             int32_t vocab, smp_dtype dtype, uint64_t seed,
                                             uint64_t offset, int32_t* out_accepted_len,
                                             int32_t* out_ids, int32_t* status, void* stream) {
  using namespace smp;
  const size_t need = smp_spec_verify_workspace_bytes(batch, k);
  if (need == 0) return SMP_ERR_INVALID_ARG;
  if (need > kStaticVerifyScratchBytes) return SMP_ERR_WORKSPACE;
  const int dev = current_device();
  if (dev < 0) return fail_cuda(cudaGetLastError());
  cudaError_t err = cudaSuccess;
  void* scratch = static_scratch_address(dev, &err);
  if (scratch == nullptr) return fail_cuda(err);
  return smp_spec_verify(p_logits, q_logits, draft_ids, batch, k, vocab, dtype, seed, offset,
                         out_accepted_len, out_ids, status, scratch, kStaticVerifyScratchBytes, stream);
}
