// Speculative-decoding verifier ("Decoding & Speculative Sampling", section
// 39.4, eqs. 39.3 and 39.4; "Speculative decoding -- Hinglish notes", section
// "The Algorithm (Step-by-Step)"; "Efficient Inference & Compression", section
// "Speculative decoding").
//
// Two kernels on the caller's stream:
//   verify_pos_kernel      one cluster per logit row (b, position, target or
//                          draft): the row maximum, the exact fixed-point mass
//                          Z and the draft token's mass, written to the
//                          workspace;
//   verify_resolve_kernel  one cluster per batch row: the accept tests in
//                          order, then the replacement draw from
//                          max(0, p_j - q_j) at the first rejection j, or the
//                          bonus draw from p_K.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"
#include "row_ops.cuh"
#include "smp.h"

namespace smp {

// Statistics of one logit row, written by verify_pos_kernel.
struct PosStat {
  float m;          // row maximum
  int32_t flags;    // kRowNonFinite / kRowBadDraft
  uint64_t z;       // sum of fixed-point masses
  double ex;        // exp(z_x - m) of the draft token (0 if none)
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
  int slice;
};

template <typename T>
__device__ __forceinline__ const T* logit_row(const VerifyArgs& a, int b, int j) {
  const size_t V = size_t(a.vocab);
  if (j <= a.k) return reinterpret_cast<const T*>(a.p) + (size_t(b) * (a.k + 1) + j) * V;
  return reinterpret_cast<const T*>(a.q) + (size_t(b) * a.k + (j - a.k - 1)) * V;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) verify_pos_kernel(VerifyArgs a) {
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  __shared__ RowShared sh;
  __shared__ FloatPair table[64];
  const uint32_t nranks = cluster_size();
  const uint32_t rank = cluster_rank();
  const int rows_per_b = 2 * a.k + 1;
  const int pr = int(blockIdx.x / nranks);
  const int b = pr / rows_per_b;
  const int j = pr % rows_per_b;
  const int V = a.vocab;
  grid_dependency_wait();
  allow_dependent_launch();
  if (threadIdx.x < 64) table[threadIdx.x] = kExp2Table[threadIdx.x];

  ClusterBarrier cbar;
  RowCtx<T> c;
  c.sh = &sh;
  c.table = table;
  c.rank = rank;
  c.nranks = nranks;
  c.first = 0;
  c.mb = 0;
  c.alive = true;
  cbar.init(&sh.mbar, &sh.ok, nranks);
  c.cb = &cbar;

  const T* row = logit_row<T>(a, b, j);
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
  int flags = 0;
  if (!key_finite<T>(key_max)) flags |= kRowNonFinite;
  const float m = key_value<T>(key_max);
  const RowScale rs = make_row_scale(m, 1.0f);
  uint64_t z = 0;
  if (!flags)
    for (int i = threadIdx.x; i < n; i += kThreads) z += mass_fixed(Elem<T>::widen(s[i]), rs, table);
  uint64_t tot[4] = {z, 0, 0, 0};
  cluster_sum4(c, tot, 1, nullptr);
  if (!c.alive) flags |= kRowTimeout;
  if (rank == 0 && threadIdx.x == 0) {
    const int i = j <= a.k ? j : j - a.k - 1;   // draft position of this row
    double ex = 0.0;
    if (i < a.k) {
      const int x = a.drafts[size_t(b) * a.k + i];
      if (x < 0 || x >= V) flags |= kRowBadDraft;
      else if (!flags) ex = mass_double(Elem<T>::widen(row[x]), rs, table);
    }
    PosStat st;
    st.m = m;
    st.flags = flags;
    st.z = tot[0];
    st.ex = ex;
    a.ws[pr] = st;
  }
  c.exchange();
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1) verify_resolve_kernel(VerifyArgs a) {
  extern __shared__ __align__(16) unsigned char dyn_smem[];
  __shared__ RowShared sh;
  __shared__ FloatPair table[64];
  __shared__ int32_t decision[2];   // first rejection j, row flags
  const uint32_t nranks = cluster_size();
  const uint32_t rank = cluster_rank();
  const int b = int(blockIdx.x / nranks);
  const int K = a.k;
  const int V = a.vocab;
  const int rows_per_b = 2 * K + 1;
  const PosStat* st = a.ws + size_t(b) * rows_per_b;
  grid_dependency_wait();   // the position statistics come from verify_pos_kernel
  allow_dependent_launch();
  if (threadIdx.x < 64) table[threadIdx.x] = kExp2Table[threadIdx.x];

  ClusterBarrier cbar;
  RowCtx<T> c;
  c.sh = &sh;
  c.table = table;
  c.rank = rank;
  c.nranks = nranks;
  c.first = 0;
  c.mb = 0;
  c.alive = true;
  cbar.init(&sh.mbar, &sh.ok, nranks);
  c.cb = &cbar;

  // Accept tests of eq. 39.3 in position order: u_i < p_i(x) / max(q_i(x), 1e-300).
  if (threadIdx.x == 0) {
    int flags = 0;
    for (int r = 0; r < rows_per_b; ++r) flags |= st[r].flags;
    int jrej = K;
    if (!flags) {
      const double scale = 1.0 / double(kFixedOne);
      for (int i = 0; i < K; ++i) {
        const PosStat& P = st[i];
        const PosStat& Q = st[K + 1 + i];
        const double p = P.ex / (double(P.z) * scale);
        const double q = Q.ex / (double(Q.z) * scale);
        const double u = double(uniform53(a.seed, a.offset, uint64_t(b), uint64_t(i))) * 0x1p-53;
        if (!(u < p / fmax(q, 1e-300))) {
          jrej = i;
          break;
        }
      }
    }
    decision[0] = jrej;
    decision[1] = flags;
  }
  __syncthreads();
  const int jrej = decision[0];
  const int flags = decision[1];

  if (flags) {
    if (rank == 0 && threadIdx.x == 0) {
      a.accepted[b] = -1;
      for (int i = 0; i <= K; ++i) a.ids[size_t(b) * (K + 1) + i] = -1;
      if (a.status) atomicOr(a.status, flags & (kRowNonFinite | kRowBadDraft | kRowTimeout));
    }
    c.exchange();
    return;
  }

  const int lo = int(rank) * a.slice;
  int n = V - lo;
  n = n < 0 ? 0 : (n > a.slice ? a.slice : n);
  c.lo = lo;
  c.n = n;
  const bool residual = jrej < K;
  const T* prow = logit_row<T>(a, b, jrej);               // p_j (or p_K for the bonus)
  const T* qrow = residual ? logit_row<T>(a, b, K + 1 + jrej) : prow;
  const PosStat P = st[jrej];
  const PosStat Q = residual ? st[K + 1 + jrej] : P;
  const size_t slice_bytes = (size_t(a.slice) * sizeof(T) + 32 + 15) & ~size_t(15);
  T* sp = reinterpret_cast<T*>(dyn_smem + slice_smem_offset(prow, lo, n));
  T* sq = reinterpret_cast<T*>(dyn_smem + slice_bytes + slice_smem_offset(qrow, lo, n));
  load_slice(prow, lo, n, sp);
  if (residual) load_slice(qrow, lo, n, sq);
  __syncthreads();
  c.s = sp;
  const RowScale rp = make_row_scale(P.m, 1.0f);
  const RowScale rq = make_row_scale(Q.m, 1.0f);

  // Weights of the final draw: max(0, p - q) scaled by Z_p Z_q (exact
  // integers, eq. 39.4), or the target masses for the bonus draw.
  bool use_p = !residual;
  auto w_res = [&](int i) -> u128 {
    const u128 ep = u128(mass_fixed(Elem<T>::widen(sp[i]), rp, table)) * Q.z;
    const u128 eq = u128(mass_fixed(Elem<T>::widen(sq[i]), rq, table)) * P.z;
    return ep > eq ? ep - eq : u128(0);
  };
  auto w_p = [&](int i) -> u128 { return u128(mass_fixed(Elem<T>::widen(sp[i]), rp, table)); };
  u128 local = 0, before = 0, total = 0;
  if (residual) {
    for (int i = threadIdx.x; i < n; i += kThreads) local += w_res(i);
    total = cluster_sum128(c, local, &before);
    if (total == 0) use_p = true;   // zero residual mass: draw from p_j
  }
  if (use_p) {
    local = 0;
    for (int i = threadIdx.x; i < n; i += kThreads) local += w_p(i);
    total = cluster_sum128(c, local, &before);
  }
  const u128 mine = block_sum<u128>(local, sh.red128);
  const uint64_t u53 = uniform53(a.seed, a.offset, uint64_t(b), uint64_t(K));
  const u128 t = scale_by_uniform(u53, total);
  if (c.alive && mine > 0 && t >= before && t - before < mine) {
    int idx;
    if (use_p)
      idx = find_crossing<T, u128>(c, t - before, w_p, sh.red128, reinterpret_cast<int*>(&sh.bcast32[7]));
    else
      idx = find_crossing<T, u128>(c, t - before, w_res, sh.red128, reinterpret_cast<int*>(&sh.bcast32[7]));
    if (threadIdx.x == 0 && idx >= 0) a.ids[size_t(b) * (K + 1) + jrej] = lo + idx;
  }
  if (rank == 0 && threadIdx.x == 0) {
    a.accepted[b] = c.alive ? jrej : -1;
    for (int i = 0; i < jrej; ++i) a.ids[size_t(b) * (K + 1) + i] = a.drafts[size_t(b) * K + i];
    for (int i = jrej + 1; i <= K; ++i) a.ids[size_t(b) * (K + 1) + i] = -1;
    if (!c.alive && a.status) atomicOr(a.status, kRowTimeout);
  }
  c.exchange();
}

// ------------------------------------------------------------------ host side

static LaunchShape verify_shape(int rows, int vocab, int elem, int num_sms, int buffers) {
  LaunchShape ls;
  int cluster = 1;
  auto slice_of = [&](int cl) { return ((vocab + cl - 1) / cl + 15) / 16 * 16; };
  while (cluster < kMaxCluster && size_t(slice_of(cluster)) * elem * buffers > kSliceTargetBytes)
    cluster *= 2;
  while (cluster < kMaxCluster && int64_t(rows) * cluster < 2 * num_sms &&
         size_t(slice_of(cluster * 2)) * elem >= kSliceMinBytes)
    cluster *= 2;
  if (forced_cluster()) cluster = forced_cluster();
  ls.cluster = cluster;
  ls.slice = slice_of(cluster);
  const size_t one = (size_t(ls.slice) * elem + 32 + 15) & ~size_t(15);
  ls.smem = one * buffers;
  ls.pdl = true;
  return ls;
}

template <typename T>
static smp_status launch_verify(VerifyArgs a, cudaStream_t stream) {
  const int dev = current_device();
  if (dev < 0) return fail_cuda(cudaGetLastError());
  const int sms = device_sms(dev);
  const int elem = int(sizeof(T));
  const int rows = a.batch * (2 * a.k + 1);
  const LaunchShape lp = verify_shape(rows, a.vocab, elem, sms, 1);
  const LaunchShape lr = verify_shape(a.batch, a.vocab, elem, sms, 2);
  if (lp.smem > kMaxDynamicSmem || lr.smem > kMaxDynamicSmem) return SMP_ERR_UNSUPPORTED;
  cudaError_t err = prepare_kernel(reinterpret_cast<const void*>(&verify_pos_kernel<T>), dev, lp);
  if (err == cudaSuccess) err = prepare_kernel(reinterpret_cast<const void*>(&verify_resolve_kernel<T>), dev, lr);
  if (err != cudaSuccess) return fail_cuda(err);
  a.slice = lp.slice;
  err = launch_cluster(reinterpret_cast<const void*>(&verify_pos_kernel<T>), dim3(rows * lp.cluster),
                       dim3(kThreads), lp, stream, &a);
  if (err != cudaSuccess) return fail_cuda(err);
  a.slice = lr.slice;
  err = launch_cluster(reinterpret_cast<const void*>(&verify_resolve_kernel<T>),
                       dim3(a.batch * lr.cluster), dim3(kThreads), lr, stream, &a);
  if (err != cudaSuccess) return fail_cuda(err);
  return SMP_OK;
}

}  // namespace smp

extern "C" size_t smp_spec_verify_workspace_bytes(int32_t batch, int32_t k) {
  if (batch <= 0 || batch > (1 << 20) || k < 1 || k > SMP_MAX_DRAFT) return 0;
  return size_t(batch) * size_t(2 * k + 1) * sizeof(smp::PosStat);
}

extern "C" smp_status smp_spec_verify(const void* p_logits, const void* q_logits,
                                      const int32_t* draft_ids, int32_t batch, int32_t k, int32_t vocab,
                                      smp_dtype dtype, uint64_t seed, uint64_t offset,
                                      int32_t* out_accepted_len, int32_t* out_ids, int32_t* status,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  using namespace smp;
  if (dtype != SMP_F32 && dtype != SMP_BF16) return SMP_ERR_DTYPE;
  if (!p_logits || !q_logits || !draft_ids || !out_accepted_len || !out_ids) return SMP_ERR_INVALID_ARG;
  if (batch <= 0 || batch > (1 << 20) || k < 1 || k > SMP_MAX_DRAFT || vocab <= 0)
    return SMP_ERR_INVALID_ARG;
  if (vocab > SMP_MAX_VOCAB) return SMP_ERR_UNSUPPORTED;
  const size_t elem = dtype == SMP_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(p_logits) % elem || reinterpret_cast<uintptr_t>(q_logits) % elem)
    return SMP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(draft_ids) % 4 || reinterpret_cast<uintptr_t>(out_ids) % 4 ||
      reinterpret_cast<uintptr_t>(out_accepted_len) % 4)
    return SMP_ERR_INVALID_ARG;
  const size_t need = smp_spec_verify_workspace_bytes(batch, k);
  if (!workspace || workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 8)
    return SMP_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (status) {
    const smp_status rc = clear_status(status, st);
    if (rc != SMP_OK) return rc;
  }
  VerifyArgs a{};
  a.p = p_logits;
  a.q = q_logits;
  a.drafts = draft_ids;
  a.batch = batch;
  a.k = k;
  a.vocab = vocab;
  a.seed = seed;
  a.offset = offset;
  a.accepted = out_accepted_len;
  a.ids = out_ids;
  a.status = status;
  a.ws = reinterpret_cast<PosStat*>(workspace);
  if (dtype == SMP_F32) return launch_verify<float>(a, st);
  return launch_verify<uint16_t>(a, st);
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
