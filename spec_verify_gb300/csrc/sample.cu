// Batched next-token sampler: temperature, top-k, top-p and min-p, the
// renormalised distribution of eq. 39.2 ("Decoding & Speculative Sampling",
// section 39.2) and an id-order inverse-CDF draw ("Choosing the next word",
// section "Where the randomness comes from, and where it stops").
//
// One thread-block cluster per row; each CTA keeps one contiguous slice of the
// row in shared memory, read from HBM exactly once.  All decisions are made on
// exact integers: logit keys for order and ties, 64-bit fixed-point masses for
// the top-p crossing and the draw, so the result does not depend on how the row
// is split or scheduled.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "launch.h"
#include "row_ops.cuh"
#include "smp.h"

namespace smp {

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
  int slice;           // elements per CTA
};

__device__ __forceinline__ bool sampling_params_valid(const smp_row_params& p) {
  const float t = p.temperature;
  if (!(isfinite(t) && t > 0.0f)) return false;
  if (p.top_k < 0) return false;
  if (isnan(p.top_p) || p.top_p < 0.0f) return false;
  if (isnan(p.min_p) || p.min_p < 0.0f) return false;
  return true;
}

template <typename T>
__device__ __forceinline__ uint32_t key_of_float(float v) {
  if (KeyTraits<T>::kBits == 32) return key_of_bits(__float_as_uint(v));
  return key_of_bits(__float_as_uint(v) & 0xFFFF0000u) >> 16;
}

// Smallest key whose value z satisfies exp((z - m) / T) >= min_p, i.e. the
// min-p threshold p_i >= min_p * max_j p_j ("Inference: Sampling, the KV
// Cache, Speculative Decoding and int8", section "Picking the next token")
// expressed on logits.  Warp 0 probes 32 keys per step, starting around the
// estimate m + T ln(min_p); every thread gets the result.
template <typename T>
__device__ uint32_t minp_threshold_key(RowShared* sh, const RowScale& rs, float temperature,
                                       float min_p, uint32_t key_max) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const double thr = double(min_p);
    const float est = rs.m + temperature * logf(min_p);
    const uint32_t k0 = key_of_float<T>(est);
    uint32_t lo = 0, hi = key_max;   // the answer lies in [lo, hi]; the property holds at hi
    uint32_t start = k0 > 16u ? k0 - 16u : 0u;
    uint32_t stride = 1;
    if (start > hi) start = hi;
    for (int iter = 0; iter < 64 && lo < hi; ++iter) {
      uint64_t cand64 = uint64_t(start) + uint64_t(lane) * stride;
      const uint32_t cand = cand64 > hi ? hi : uint32_t(cand64);
      const bool ok = mass_double(key_value<T>(cand), rs, sh->table) >= thr;
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
    if (lane == 0) sh->bcast32[6] = hi;
  }
  __syncthreads();
  const uint32_t r = sh->bcast32[6];
  __syncthreads();
  return r;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) sample_kernel(SampleArgs a) {
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  __shared__ RowShared sh;
  const uint32_t nranks = cluster_size();
  const uint32_t rank = cluster_rank();
  const int b = int(blockIdx.x / nranks);
  const int V = a.vocab;
  if (threadIdx.x < 64) sh.table[threadIdx.x] = kExp2Table[threadIdx.x];

  RowCtx<T> c;
  c.sh = &sh;
  c.rank = rank;
  c.nranks = nranks;
  c.mb = 0;
  c.alive = true;
  c.cb.init(&sh.mbar, &sh.ok, nranks);

  const T* row = reinterpret_cast<const T*>(a.logits) + size_t(b) * size_t(V);
  const int lo = int(rank) * a.slice;
  int n = V - lo;
  n = n < 0 ? 0 : (n > a.slice ? a.slice : n);
  c.lo = lo;
  c.n = n;
  T* s = reinterpret_cast<T*>(dyn_smem + slice_smem_offset(row, lo, n));
  c.s = s;

  uint64_t best = load_slice(row, lo, n, s);
  __syncthreads();
  best = cluster_max(c, best);
  const uint32_t key_max = uint32_t(best >> 32);
  const uint32_t argmax = ~uint32_t(best);
  const smp_row_params prm = a.params[b];
  const bool greedy = prm.greedy != 0 || prm.temperature == 0.0f;

  int flags = 0;
  if (!c.alive) flags |= kRowTimeout;
  else if (!key_finite<T>(key_max)) flags |= kRowNonFinite;
  else if (!greedy && !sampling_params_valid(prm)) flags |= kRowBadParams;

  if (flags == 0 && greedy) {
    if (rank == 0 && threadIdx.x == 0) {
      a.out_ids[b] = int32_t(argmax);
      if (a.out_probs) a.out_probs[b] = 1.0f;
      if (a.kept) a.kept[b] = 1;
    }
    if (a.full_probs) {
      float* f = a.full_probs + size_t(b) * V + lo;
      for (int i = threadIdx.x; i < n; i += kThreads) f[i] = (uint32_t(lo + i) == argmax) ? 1.0f : 0.0f;
    }
    c.exchange();
    return;
  }

  if (flags == 0) {
    const float m = key_value<T>(key_max);
    const RowScale rs = make_row_scale(m, prm.temperature);
    const bool topk = prm.top_k > 0 && prm.top_k < V;
    const bool topp = prm.top_p < 1.0f;
    const bool minp = prm.min_p > 0.0f && prm.min_p < 1.0f;
    uint32_t key_min_p = 0;
    if (minp) key_min_p = minp_threshold_key<T>(&sh, rs, prm.temperature, prm.min_p, key_max);

    // Row statistics: size of the min-p set and the total mass Z.
    uint64_t stats[4] = {0, 0, 0, 0};
    if (minp || topp) {
      uint64_t cnt = 0, z = 0;
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const T v = s[i];
        if (minp && elem_key<T>(v) >= key_min_p) ++cnt;
        if (topp) z += mass_fixed(Elem<T>::widen(v), rs, sh.table);
      }
      stats[0] = cnt;
      stats[1] = z;
      cluster_sum4(c, stats, 2, nullptr);
    }
    const uint64_t len_m = minp ? stats[0] : uint64_t(V);
    const uint64_t z_total = stats[1];

    Boundary bk{}, bp{};
    uint64_t len_k = uint64_t(V), len_p = uint64_t(V);
    if (topk) {
      bk = radix_select<T, false>(c, uint32_t(prm.top_k), MassTarget{}, rs);
      len_k = uint64_t(prm.top_k);
    }
    if (topp) {
      const MassTarget tgt = make_mass_target(prm.top_p, z_total);
      bp = radix_select<T, true>(c, 0, tgt, rs);
      len_p = uint64_t(bp.above) + bp.n;
    }
    // The kept set is the shortest of the prefixes (eq. 39.2 on the
    // intersection of the masks).
    uint64_t len = len_k < len_p ? len_k : len_p;
    len = len < len_m ? len : len_m;
    int mode = 0;   // 0: all; 1: key >= key_min_p; 2: boundary (key, id_cut)
    Boundary bd{};
    if (len < uint64_t(V)) {
      if (minp && len == len_m) mode = 1;
      else {
        mode = 2;
        bd = (topk && len == len_k) ? bk : bp;
      }
    }
    uint32_t id_cut = 0xFFFFFFFFu;
    if (mode == 2 && bd.n < bd.tie_total) {
      uint32_t mine = 0xFFFFFFFFu;
      if (bd.n > bd.tie_base && bd.n <= bd.tie_base + bd.tie_local)
        mine = nth_with_key(c, bd.key, bd.n - bd.tie_base);
      id_cut = cluster_min_id(c, mine);
    }
    auto kept = [&](int i) -> bool {
      if (mode == 0) return true;
      const uint32_t key = elem_key<T>(s[i]);
      if (mode == 1) return key >= key_min_p;
      return key > bd.key || (key == bd.key && uint32_t(lo + i) <= id_cut);
    };
    auto weight = [&](int i) -> uint64_t {
      return kept(i) ? mass_fixed(Elem<T>::widen(s[i]), rs, sh.table) : 0ull;
    };

    // Kept mass Z_S of this CTA, of the row, and the prefix over CTAs.
    uint64_t zs = 0;
    for (int i = threadIdx.x; i < n; i += kThreads) zs += weight(i);
    uint64_t tot[4] = {zs, 0, 0, 0};
    uint64_t z_before = 0, z_local = 0;
    cluster_sum4(c, tot, 1, &z_before, &z_local);
    const uint64_t z_kept = tot[0];

    // The draw: the first kept token (id order) whose running mass exceeds
    // t = floor(u * Z_S), u = Philox draw 0 of row b.
    const uint64_t u53 = uniform53(a.seed, a.offset, uint64_t(b), 0);
    const uint64_t t = uint64_t((u128(u53) * z_kept) >> 53);
    if (c.alive && z_local > 0 && t >= z_before && t - z_before < z_local) {
      const int idx = find_crossing<T, uint64_t>(c, t - z_before, weight, sh.red64,
                                                 reinterpret_cast<int*>(&sh.bcast32[7]));
      if (threadIdx.x == 0 && idx >= 0) {
        const uint64_t e = weight(idx);
        a.out_ids[b] = lo + idx;
        if (a.out_probs) a.out_probs[b] = float(double(e) / double(z_kept));
      }
    }
    if (a.kept && rank == 0 && threadIdx.x == 0) a.kept[b] = int32_t(len);
    if (a.full_probs) {
      float* f = a.full_probs + size_t(b) * V + lo;
      const float zf = float(z_kept);
      for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint64_t e = weight(i);
        f[i] = e ? __fdiv_rn(float(e), zf) : 0.0f;
      }
    }
    if (!c.alive) flags |= kRowTimeout;
  }

  if (flags) {
    if (rank == 0 && threadIdx.x == 0) {
      a.out_ids[b] = -1;
      if (a.out_probs) a.out_probs[b] = __int_as_float(0x7FC00000);
      if (a.kept) a.kept[b] = 0;
      if (a.status) atomicOr(a.status, flags);
    }
    if (a.full_probs && !(flags & kRowTimeout)) {
      float* f = a.full_probs + size_t(b) * V + lo;
      for (int i = threadIdx.x; i < n; i += kThreads) f[i] = __int_as_float(0x7FC00000);
    }
  }
  c.exchange();   // no CTA leaves while a peer may still read its mailboxes
}

// ------------------------------------------------------------------ host side

// Shape of the launch for a row of `vocab` elements of `elem` bytes.
static LaunchShape sample_shape(int batch, int vocab, int elem, int num_sms) {
  LaunchShape ls;
  int cluster = 1;
  auto slice_of = [&](int cl) { return ((vocab + cl - 1) / cl + 15) / 16 * 16; };
  while (cluster < kMaxCluster && size_t(slice_of(cluster)) * elem > kSliceTargetBytes) cluster *= 2;
  while (cluster < kMaxCluster && int64_t(batch) * cluster < 2 * num_sms &&
         size_t(slice_of(cluster * 2)) * elem >= kSliceMinBytes)
    cluster *= 2;
  if (forced_cluster()) cluster = forced_cluster();
  ls.cluster = cluster;
  ls.slice = slice_of(cluster);
  ls.smem = size_t(ls.slice) * elem + 32;
  return ls;
}

template <typename T>
static smp_status launch_sample(const SampleArgs& args, int elem, cudaStream_t stream) {
  const int dev = current_device();
  if (dev < 0) return fail_cuda(cudaGetLastError());
  const LaunchShape ls = sample_shape(args.batch, args.vocab, elem, device_sms(dev));
  if (ls.smem > kMaxDynamicSmem) return SMP_ERR_UNSUPPORTED;
  SampleArgs a = args;
  a.slice = ls.slice;
  cudaError_t err = prepare_kernel(reinterpret_cast<const void*>(&sample_kernel<T>), dev, ls);
  if (err != cudaSuccess) return fail_cuda(err);
  err = launch_cluster(reinterpret_cast<const void*>(&sample_kernel<T>), dim3(args.batch * ls.cluster),
                       dim3(kThreads), ls, stream, &a);
  if (err != cudaSuccess) return fail_cuda(err);
  return SMP_OK;
}

static smp_status sample_common(const void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                                const smp_row_params* params, uint64_t seed, uint64_t offset,
                                int32_t* out_ids, float* out_probs, float* full, int32_t* kept,
                                int32_t* status, void* stream) {
  if (dtype != SMP_F32 && dtype != SMP_BF16) return SMP_ERR_DTYPE;
  if (!logits || !params || !out_ids) return SMP_ERR_INVALID_ARG;
  if (batch <= 0 || vocab <= 0) return SMP_ERR_INVALID_ARG;
  if (vocab > SMP_MAX_VOCAB) return SMP_ERR_UNSUPPORTED;
  const int elem = dtype == SMP_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(logits) % elem) return SMP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(params) % 4 || reinterpret_cast<uintptr_t>(out_ids) % 4)
    return SMP_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (status) {
    const cudaError_t err = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    if (err != cudaSuccess) return fail_cuda(err);
  }
  SampleArgs a{};
  a.logits = logits;
  a.batch = batch;
  a.vocab = vocab;
  a.params = params;
  a.seed = seed;
  a.offset = offset;
  a.out_ids = out_ids;
  a.out_probs = out_probs;
  a.status = status;
  a.full_probs = full;
  a.kept = kept;
  if (dtype == SMP_F32) return launch_sample<float>(a, 4, st);
  return launch_sample<uint16_t>(a, 2, st);
}

}  // namespace smp

extern "C" smp_status smp_sample(const void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                                 const smp_row_params* params, uint64_t seed, uint64_t offset,
                                 int32_t* out_ids, float* out_probs, int32_t* status, void* stream) {
  return smp::sample_common(logits, batch, vocab, dtype, params, seed, offset, out_ids, out_probs,
                            nullptr, nullptr, status, stream);
}

extern "C" smp_status smp_filter_debug(const void* logits, int32_t batch, int32_t vocab,
                                       smp_dtype dtype, const smp_row_params* params, uint64_t seed,
                                       uint64_t offset, int32_t* out_ids, float* out_probs,
                                       float* out_probs_full, int32_t* out_kept, int32_t* status,
                                       void* stream) {
  if (!out_probs_full || !out_kept) return SMP_ERR_INVALID_ARG;
  return smp::sample_common(logits, batch, vocab, dtype, params, seed, offset, out_ids, out_probs,
                            out_probs_full, out_kept, status, stream);
}
