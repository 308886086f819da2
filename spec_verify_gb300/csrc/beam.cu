// One beam-search step's candidate selection ("Decoding & Speculative
// Sampling", section 39.1, eq. 39.1 and Listing 39.1; "Efficient Inference &
// Compression", section "Beam search"): every beam b of a group is extended
// by every token t with score s_b + log p_b(t), and the `width` best of the
// group's beams x V candidates survive, ordered by score (equal scores: lower
// flat index b * V + t first).
//
// Two kernels on the caller's stream:
//   beam_row_kernel    one CTA per slice of a beam row: the slice maximum,
//                      its mass sum (binary32 exponentials, fixed-point
//                      sums), and its `width` best tokens by (logit desc,
//                      id asc): the elements at or above the width-th
//                      largest thread maximum, ranked exactly (the sampler's
//                      radix selection when too many tie there);
//   beam_merge_kernel  one CTA per group: each beam's m and Z from its
//                      slices, the scores s_b + (z - m_b - ln Z_b) in fp64 of
//                      the listed tokens, and the group's best `width` of
//                      them, picked by warp 0 in rounds of reductions,
//                      written in rank order.
// Only a row's best `width` tokens can be among its group's best `width`
// candidates, because within a beam the score order is the logit order.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>

#include "launch.h"
#include "row_ops.cuh"
#include "smp.h"

namespace smp {

#include "select.cuh"

// Each beam row is cut into S slices of about V / S ids, one CTA per slice,
// so that a few rows still spread over the GPU.  Per slice in the workspace:
// its header, then `width` (id, logit) pairs, its best tokens by (logit desc,
// id asc).  The union of a row's slice lists holds the row's best `width`.
constexpr int kBeamMaxSlices = 16;
constexpr int kBeamU = 8;   // 16-byte loads in flight per thread in the slice passes
constexpr int kBeamMaxCand = SMP_MAX_BEAM_WIDTH * SMP_MAX_BEAM_WIDTH;   // candidates one merge CTA ranks
constexpr int kSliceEmpty = 1 << 8;   // a slice with no finite logit (not an error by itself)

struct BeamSliceHead {
  float m;         // the slice's maximum logit
  int32_t flags;   // kSliceEmpty, or kRowNonFinite (+inf in the slice)
  uint64_t z;      // sum of exp(z - m) over the slice, 44-bit fixed point
  int32_t n;       // candidates listed
  int32_t pad;
};
struct BeamCand {
  int32_t id;
  float z;
};

struct BeamArgs {
  const void* logits;   // [groups, beams, vocab]
  const double* scores; // [groups, beams]
  int groups;
  int beams;
  int vocab;
  int width;
  int slices;           // S
  int slice_len;        // ids per slice (a multiple of 8)
  int32_t* out_parent;  // [groups, width]
  int32_t* out_token;
  double* out_score;
  int32_t* status;
  unsigned char* ws;
};

__host__ __device__ __forceinline__ size_t beam_slice_bytes(int width) {
  return sizeof(BeamSliceHead) + size_t(width) * sizeof(BeamCand);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2) beam_row_kernel(BeamArgs a) {
  __shared__ FloatPair table[64];
  __shared__ GenShared gs;
  __shared__ unsigned long long members[SMP_MAX_BEAM_WIDTH];   // (key << 32) | ~local id
  __shared__ int n_members;
  const int tid = threadIdx.x;
  const int rowi = int(blockIdx.x) / a.slices;
  const int slice = int(blockIdx.x) % a.slices;
  grid_dependency_wait();
  allow_dependent_launch();
  if (tid < 64) table[tid] = kExp2Table[tid];
  if (tid == 0) n_members = 0;
  const int lo = slice * a.slice_len;
  const int len = max(0, min(a.vocab, lo + a.slice_len) - lo);
  const T* row = reinterpret_cast<const T*>(a.logits) + size_t(rowi) * a.vocab + lo;
  BeamSliceHead* head = reinterpret_cast<BeamSliceHead*>(a.ws + size_t(blockIdx.x) * beam_slice_bytes(a.width));
  BeamCand* cand = reinterpret_cast<BeamCand*>(head + 1);
  if (len == 0) {
    if (tid == 0) {
      head->m = -INFINITY;
      head->flags = kSliceEmpty;
      head->z = 0;
      head->n = 0;
    }
    return;
  }

  // One pass for the slice maximum and Z = sum exp(z - m): each thread keeps
  // a running maximum tm and the binary32 sum st of exp(z - tm) over its
  // elements, rescaled when a group of kBeamU vectors raises tm; its share,
  // scaled to the slice maximum, is turned into 44-bit fixed point once and
  // summed exactly.  NaN counts as -inf (the packed maxima skip it, and its
  // exponential is 0).
  using Vo = VecOps<T>;
  constexpr int kPer = Vo::kPer;
  const RowScale unit = make_row_scale_unit(0.0f);
  float tm = -INFINITY, st = 0.0f;
  auto raise_to = [&](float g) {   // g > tm
    st = tm > -INFINITY ? __fmul_rn(st, exp_fast(tm, RowScale{g, unit.c_hi, unit.c_lo})) : 0.0f;
    tm = g;
  };
  {
    const uintptr_t r0 = reinterpret_cast<uintptr_t>(row);
    const uintptr_t a0 = (r0 + 15) & ~uintptr_t(15), a1 = (r0 + size_t(len) * sizeof(T)) & ~uintptr_t(15);
    const bool mid = a1 > a0;
    const int head = mid ? int((a0 - r0) / sizeof(T)) : len;
    const int tail0 = mid ? int((a1 - r0) / sizeof(T)) : len;
    const int nvec = mid ? int((a1 - a0) / 16) : 0;
    const uint4* vp = reinterpret_cast<const uint4*>(a0);
    const uint32_t ninf = Vo::neg_inf();
    for (int v0 = tid; v0 < nvec; v0 += kThreads * kBeamU) {
      uint4 x[kBeamU];
      uint32_t pm = ninf;
#pragma unroll
      for (int u = 0; u < kBeamU; ++u) {
        x[u] = v0 + u * kThreads < nvec ? __ldg(vp + v0 + u * kThreads) : make_uint4(ninf, ninf, ninf, ninf);
        pm = Vo::max2(pm, Vo::vmax(x[u]));
      }
      const float gmx = Vo::finish(pm);
      if (gmx > tm) raise_to(gmx);
      if (tm > -INFINITY) {
        const RowScale rt{tm, unit.c_hi, unit.c_lo};
        float acc = 0.0f;
#pragma unroll
        for (int u = 0; u < kBeamU; ++u)
#pragma unroll
          for (int q = 0; q < kPer; ++q) acc += exp_fast(Vo::elem(x[u], q), rt);
        st += acc;
      }
    }
    auto edge = [&](float z) {
      if (z > tm) raise_to(z);
      if (tm > -INFINITY) st += exp_fast(z, RowScale{tm, unit.c_hi, unit.c_lo});
    };
    for (int i = tid; i < head; i += kThreads) edge(Elem<T>::widen(row[i]));
    for (int i = tail0 + tid; i < len; i += kThreads) edge(Elem<T>::widen(row[i]));
  }
  const uint32_t kmine = order_key<T>(tm);   // this thread's maximum key
  const uint32_t kmax = uint32_t(block_max_u64(uint64_t(kmine), gs.red64));
  if (!key_finite<T>(kmax)) {   // all -inf / NaN, or +inf present
    if (tid == 0) {
      const bool pinf = kmax == order_key<T>(INFINITY);
      head->m = -INFINITY;
      head->flags = pinf ? kRowNonFinite : kSliceEmpty;
      head->z = 0;
      head->n = 0;
    }
    return;
  }
  const float m = key_value<T>(kmax);
  const RowScale rs = make_row_scale_unit(m);
  const float share = tm > -INFINITY ? __fmul_rn(st, exp_fast(tm, rs)) : 0.0f;
  uint64_t zf = __float2ull_rn(__fmul_rn(share, float(kFixedOne)));
  zf = warp_sum<uint64_t>(zf);
  if ((tid & 31) == 0) gs.scan64[tid >> 5] = zf;

  // The slice's `width` best tokens by (key desc, id asc).  theta = the
  // width-th largest of the threads' maxima: at least `width` elements reach
  // it, so every one of the best `width` does.  The elements >= theta are
  // listed and ranked exactly; if there are too many (many equal logits),
  // the exact radix selection of the sampler finds the boundary instead.
  // theta = the kw-th largest of the threads' maxima (a multiset): each warp
  // lists its kw largest lane maxima by repeated warp maxima, then warp 0 takes
  // the kw-th largest of the warps' lists the same way.  Real keys are above 0.
  const int kw = min(a.width, len);
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t* wtop = &gs.cnt[0][0];   // kWarps * kw keys
  {
    bool in = true;
    for (int r = 0; r < kw; ++r) {
      const uint32_t mx = __reduce_max_sync(0xFFFFFFFFu, in ? kmine : 0u);
      const uint32_t who = __ballot_sync(0xFFFFFFFFu, in && kmine == mx);
      if (lane == __ffs(who) - 1) in = false;
      if (lane == 0) wtop[warp * kw + r] = mx;
    }
  }
  cta_sync();
  uint64_t ztot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) ztot += gs.scan64[w];
  if (warp == 0) {
    constexpr int kPerLane = kWarps * SMP_MAX_BEAM_WIDTH / 32;
    const int total = kWarps * kw;
    uint32_t v[kPerLane];
    uint32_t act = 0;   // bit j: v[j] still in the multiset
#pragma unroll
    for (int j = 0; j < kPerLane; ++j) {
      const int idx = lane + 32 * j;
      v[j] = idx < total ? wtop[idx] : 0u;
      act |= (idx < total ? 1u : 0u) << j;
    }
    uint32_t kth = 0;
    for (int r = 0; r < kw; ++r) {
      uint32_t lm = 0;
      int lj = -1;
#pragma unroll
      for (int j = 0; j < kPerLane; ++j)
        if (((act >> j) & 1u) && (lj < 0 || v[j] > lm)) {
          lm = v[j];
          lj = j;
        }
      kth = __reduce_max_sync(0xFFFFFFFFu, lj >= 0 ? lm : 0u);
      const uint32_t who = __ballot_sync(0xFFFFFFFFu, lj >= 0 && lm == kth);
      if (lane == __ffs(who) - 1) act &= ~(1u << lj);
    }
    if (lane == 0) gs.bc32[0] = kth;
  }
  cta_sync();
  const uint32_t theta = gs.bc32[0];
  unsigned long long* list = reinterpret_cast<unsigned long long*>(&gs.mass[0][0][0]);   // kBeamList entries
  constexpr int kBeamList = int(sizeof(gs.mass) / sizeof(unsigned long long));
  if (tid == 0) n_members = 0;
  cta_sync();
  // A finite theta: the sampler's candidate pass (a bit per element, one
  // atomic per warp, the marked logits read again), up to kTopCandMax
  // entries; else (NaN counts as -inf, and -inf may be listed) one atomic
  // per listed element, up to kBeamList.
  const bool finite_theta = key_finite<T>(theta);
  if (finite_theta) {
    topk_candidate_pass<T, kBeamU, true, false>(row, len, theta, key_value<T>(theta), RowScale{}, list,
                                                reinterpret_cast<uint32_t*>(&n_members), NoPrep());
  } else {
    gen_sweep<T, kBeamU>(row, len, [&](int i, float z) {
      const uint32_t k = order_key<T>(z);   // NaN has the key of -inf
      if (k >= theta) {
        const int slot = atomicAdd(&n_members, 1);
        if (slot < kBeamList) list[slot] = pack_key_id(k, uint32_t(i));
      }
    });
  }
  cta_sync();
  int nl = n_members;
  if (nl > (finite_theta ? kTopCandMax : kBeamList)) {   // too many at or above theta: exact radix selection of the boundary
    smp_row_params prm;
    prm.temperature = 1.0f;
    prm.top_k = a.width;
    prm.top_p = 1.0f;
    prm.min_p = 0.0f;
    prm.greedy = 0;
    cta_sync();
    const KeptSet ks = gen_kept_set<T>(row, len, gs, table, prm, kmax);
    if (tid == 0) n_members = 0;
    cta_sync();
    gen_sweep<T>(row, len, [&](int i, float z) {
      const uint32_t k = order_key<T>(isnan(z) ? -INFINITY : z);
      if (in_kept_set(ks, k, uint32_t(i))) {
        const int slot = atomicAdd(&n_members, 1);
        if (slot < SMP_MAX_BEAM_WIDTH) members[slot] = pack_key_id(k, uint32_t(i));
      }
    });
    cta_sync();
    nl = min(n_members, SMP_MAX_BEAM_WIDTH);
    list = members;
  }
  // The listed values ranked in decreasing order; the first kw are kept.
  for (int c = tid; c < nl; c += kThreads) {
    const unsigned long long mine = list[c];
    int rank = 0;
    for (int j = 0; j < nl && rank < kw; ++j) rank += list[j] > mine;
    if (rank < kw) {
      const uint32_t id = ~uint32_t(mine);
      const float z = Elem<T>::widen(row[id]);
      cand[rank].id = lo + int32_t(id);
      cand[rank].z = isnan(z) ? -INFINITY : z;
    }
  }
  if (tid == 0) {
    head->m = m;
    head->flags = 0;
    head->z = ztot;
    head->n = min(kw, nl);
  }
}

// ln z for z >= 1: the binary32 logarithm (logf) of z's mantissa in [1, 2),
// plus its exponent times ln 2 in fp64.  The mantissa's rounding to binary32
// and logf each add at most about 6e-8 (absolute; ln of the mantissa < 0.7).
__device__ __forceinline__ double ln_of_sum(double z) {
  const long long bits = __double_as_longlong(z);
  const int e = int((bits >> 52) & 0x7FF) - 1023;
  const double mant = __longlong_as_double((bits & 0x000FFFFFFFFFFFFFll) | 0x3FF0000000000000ll);
  return double(logf(float(mant))) + double(e) * 0.6931471805599453;
}

// One CTA per group.  Per beam: m = the slices' maximum, Z = sum over slices
// of Z_s exp(m_s - m) (binary32 exponentials, fp64 products and sums),
// c = -m - ln Z.  Every listed candidate gets its score s_b + (z + c_b) and
// its flat index b * V + id; in the order (score desc, flat asc), a strict
// total order, the first `width` are picked one per round and written at
// their ranks.
__global__ void __launch_bounds__(kThreads) beam_merge_kernel(BeamArgs a) {
  __shared__ double cs[kBeamMaxCand];
  __shared__ int32_t cf[kBeamMaxCand];   // flat index, or -1 for an empty slot
  __shared__ double beam_c[SMP_MAX_BEAM_WIDTH];
  __shared__ float beam_m[SMP_MAX_BEAM_WIDTH];
  __shared__ int beam_f[SMP_MAX_BEAM_WIDTH];
  __shared__ int bad;
  const int g = int(blockIdx.x);
  const int W = a.beams, width = a.width, V = a.vocab, S = a.slices;
  const int tid = threadIdx.x;
  grid_dependency_wait();
  allow_dependent_launch();
  auto head_of = [&](int b, int s) {
    return reinterpret_cast<const BeamSliceHead*>(a.ws + (size_t(g * W + b) * S + s) * beam_slice_bytes(width));
  };
  if (tid == 0) bad = 0;
  // The slice headers, one load per thread and all in flight at once, staged
  // in the candidate arrays (free until the candidates are built): Z_s in
  // cs[c], the flags in cf[c], the bits of m_s in cf[half + c] (W * S <= half).
  constexpr int kHalf = kBeamMaxCand / 2;
  for (int c = tid; c < W * S; c += kThreads) {
    const BeamSliceHead* h = head_of(c / S, c % S);
    cs[c] = double(h->z) * (1.0 / double(kFixedOne));
    cf[kHalf + c] = __float_as_int(h->m);
    cf[c] = h->flags;
  }
  __syncthreads();
  // Per beam (thread b): the flags and the slices' maximum m.
  if (tid < W) {
    const int b = tid;
    int f = isnan(a.scores[size_t(g) * W + b]) ? kRowBadParams : 0;
    float m = -INFINITY;   // the slices' maxima are binary32 logits: fp32 operations, exact
    bool any = false;
    for (int s = 0; s < S; ++s) {
      const int fl = cf[b * S + s];
      f |= fl & kRowNonFinite;
      if (!fl) {
        any = true;
        m = fmaxf(m, __int_as_float(cf[kHalf + b * S + s]));
      }
    }
    if (!any) f |= kRowNonFinite;
    beam_m[b] = m;
    beam_f[b] = f;
    if (f) atomicOr(&bad, f);
  }
  __syncthreads();
  // Each slice's Z_s exp(m_s - m), one per thread: the binary32 exponential
  // (expf) of the binary32 difference, times Z_s in fp64.  The fp64 pipe of
  // this part is narrow, so the merge keeps fp64 to sums and products.
  for (int c = tid; c < W * S; c += kThreads) {
    const int b = c / S;
    cs[c] = (beam_f[b] || cf[c]) ? 0.0 : cs[c] * double(expf(__fsub_rn(__int_as_float(cf[kHalf + c]), beam_m[b])));
  }
  __syncthreads();
  if (tid < W) {   // Z in slice order, then the beam's constant -m - ln Z
    const int b = tid;
    double z = 0.0;
    if (!beam_f[b])
      for (int s = 0; s < S; ++s)
        if (!cf[b * S + s]) z += cs[b * S + s];
    beam_c[b] = beam_f[b] ? 0.0 : -double(beam_m[b]) - ln_of_sum(z);
  }
  // ranks nobody fills (fewer candidates than width, or an error group) stay -1 / NaN
  for (int r = tid; r < width; r += kThreads) {
    a.out_parent[size_t(g) * width + r] = -1;
    a.out_token[size_t(g) * width + r] = -1;
    a.out_score[size_t(g) * width + r] = __longlong_as_double(0x7FF8000000000000ll);
  }
  __syncthreads();
  if (bad) {
    if (tid == 0 && a.status) atomicOr(a.status, bad);
    return;
  }
  const int per_beam = S * width;
  const int n = W * per_beam;
  for (int c = tid; c < n; c += kThreads) {
    const int b = c / per_beam, s = (c % per_beam) / width, j = c % width;
    const BeamSliceHead* h = head_of(b, s);
    cf[c] = -1;
    cs[c] = 0.0;
    if (j < h->n) {
      const BeamCand* l = reinterpret_cast<const BeamCand*>(h + 1);
      cs[c] = a.scores[size_t(g) * W + b] + (double(l[j].z) + beam_c[b]);
      cf[c] = b * V + l[j].id;
    }
  }
  // The scores as order keys in place (the fp64 bits with the sign folded
  // in, -0 as +0), so that the rank loop compares integers: fp64 comparisons
  // run on the narrow fp64 pipe of this part.
  auto to_key = [](double x) -> unsigned long long {
    const unsigned long long b = (unsigned long long)__double_as_longlong(x == 0.0 ? 0.0 : x);
    return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
  };
  auto from_key = [](unsigned long long k) -> double {
    return __longlong_as_double((long long)((k >> 63) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k));
  };
  unsigned long long* ck = reinterpret_cast<unsigned long long*>(cs);
  __syncthreads();
  for (int c = tid; c < n; c += kThreads) ck[c] = to_key(cs[c]);
  __syncthreads();
  // The best `width` in rounds, by warp 0 alone: each round every lane
  // offers its best candidate not yet taken (score key desc, flat asc), a
  // warp reduction picks the round's winner, written at that rank and taken.
  // (A rank per candidate by comparison with all others ran one shared load
  // after another, 8-11 us for 144 candidates; rounds with CTA barriers
  // took about 3 us.)
  if (tid < 32) {
    const int lane = tid;
    for (int r = 0; r < width; ++r) {
      unsigned long long bk = 0;
      int bf = INT_MAX, bc = -1;
      for (int c = lane; c < n; c += 32) {
        const int f = cf[c];
        if (f < 0) continue;
        const unsigned long long k = ck[c];
        if (bc < 0 || k > bk || (k == bk && f < bf)) {
          bk = k;
          bf = f;
          bc = c;
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const unsigned long long ok = shfl_xor_u64(bk, o);
        const int of = __shfl_xor_sync(0xFFFFFFFFu, bf, o);
        const int oc = __shfl_xor_sync(0xFFFFFFFFu, bc, o);
        if (oc >= 0 && (bc < 0 || ok > bk || (ok == bk && of < bf))) {
          bk = ok;
          bf = of;
          bc = oc;
        }
      }
      if (bc < 0) break;   // none left (every lane agrees): the remaining ranks keep -1 / NaN
      if (lane == 0) {
        a.out_parent[size_t(g) * width + r] = bf / V;
        a.out_token[size_t(g) * width + r] = bf % V;
        a.out_score[size_t(g) * width + r] = from_key(bk);
        cf[bc] = -1;
      }
      __syncwarp();
    }
  }
}

template <typename T>
static smp_status launch_beam(const BeamArgs& args, cudaStream_t stream) {
  BeamArgs a = args;
  const int dev = current_device();
  if (dev < 0) return fail_cuda(cudaGetLastError());
  // Slices: as many CTAs as fit in one wave at two per SM (rounded down, so
  // that no slice waits for a second wave), at most kBeamMaxSlices, at least
  // 2048 ids each, and no more candidates per group than one merge CTA ranks.
  const int64_t rows = int64_t(a.groups) * a.beams;
  int S = int(2 * int64_t(device_sms(dev)) / rows);
  S = std::min(S, kBeamMaxSlices);
  S = std::min(S, kBeamMaxCand / (a.beams * a.width));
  S = std::min(S, (a.vocab + 2047) / 2048);
  S = std::max(S, 1);
  a.slices = S;
  a.slice_len = ((a.vocab + S - 1) / S + 7) / 8 * 8;
  LaunchShape ls;
  ls.pdl = true;
  cudaError_t err = launch_cluster(reinterpret_cast<const void*>(&beam_row_kernel<T>),
                                   dim3(unsigned(rows * S)), dim3(kThreads), ls, stream, &a);
  if (err != cudaSuccess) return fail_cuda(err);
  err = launch_cluster(reinterpret_cast<const void*>(&beam_merge_kernel), dim3(unsigned(a.groups)), dim3(kThreads),
                       ls, stream, &a);
  if (err != cudaSuccess) return fail_cuda(err);
  return SMP_OK;
}

}  // namespace smp

extern "C" size_t smp_beam_topk_workspace_bytes(int32_t groups, int32_t beams, int32_t width) {
  if (groups <= 0 || beams <= 0 || width <= 0 || width > SMP_MAX_BEAM_WIDTH || beams > SMP_MAX_BEAM_WIDTH ||
      int64_t(groups) * beams > (1 << 24))
    return 0;
  return size_t(groups) * size_t(beams) * smp::kBeamMaxSlices * smp::beam_slice_bytes(width);
}

extern "C" smp_status smp_beam_topk(const void* logits, const double* beam_scores, int32_t groups, int32_t beams,
                                    int32_t vocab, int32_t width, smp_dtype dtype, int32_t* out_parent,
                                    int32_t* out_token, double* out_score, int32_t* status, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  using namespace smp;
  if (dtype != SMP_F32 && dtype != SMP_BF16) return SMP_ERR_DTYPE;
  if (!logits || !beam_scores || !out_parent || !out_token || !out_score) return SMP_ERR_INVALID_ARG;
  if (vocab <= 0 || int64_t(beams) * vocab > INT_MAX) return SMP_ERR_INVALID_ARG;
  const size_t need = smp_beam_topk_workspace_bytes(groups, beams, width);
  if (need == 0) return SMP_ERR_INVALID_ARG;
  if (vocab > SMP_MAX_VOCAB) return SMP_ERR_UNSUPPORTED;
  const int elem = dtype == SMP_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(logits) % elem || reinterpret_cast<uintptr_t>(beam_scores) % 8 ||
      reinterpret_cast<uintptr_t>(out_score) % 8 ||
      (reinterpret_cast<uintptr_t>(out_parent) | reinterpret_cast<uintptr_t>(out_token) |
       reinterpret_cast<uintptr_t>(status)) % 4)
    return SMP_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 8) return SMP_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (status) {
    const smp_status rc = clear_status(status, st);
    if (rc != SMP_OK) return rc;
  }
  BeamArgs a{};
  a.logits = logits;
  a.scores = beam_scores;
  a.groups = groups;
  a.beams = beams;
  a.vocab = vocab;
  a.width = width;
  a.out_parent = out_parent;
  a.out_token = out_token;
  a.out_score = out_score;
  a.status = status;
  a.ws = reinterpret_cast<unsigned char*>(workspace);
  if (dtype == SMP_F32) return launch_beam<float>(a, st);
  return launch_beam<uint16_t>(a, st);
}
