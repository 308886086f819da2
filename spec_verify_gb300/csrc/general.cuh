// General path of the sampler: any knobs (top-p, unfiltered sampling, any k,
// and rows whose candidates overflow), exactly, by one CTA per row over the
// row in global memory ("Decoding & Speculative Sampling", section 39.2 and
// eq. 39.2; "Choosing the next word", section "Where the randomness comes
// from, and where it stops").
//
// The kept set, the shortest of the enabled prefixes of the order (logit
// descending, id ascending), comes from gen_kept_set (select.cuh), by radix
// selection over order keys, or, for top-k up to kTopKMax, from
// gen_kept_set_topk's ranked candidate list, which the draw then reads in
// place of a walk over the row.  Included by sample.cu
// inside namespace smp, after the sampler's argument block and row helpers
// it uses.
#pragma once

// The draw over a kept set held as a list (topk_list and topk_mass, len
// entries in rank order): the token whose interval [run, run + E) of the
// running mass in id order holds t.  Each of the first len threads sums the
// masses of the listed tokens with lower ids.
__device__ __forceinline__ int topk_draw(GenShared& gs, uint32_t len, uint64_t t) {
  const unsigned long long* list = topk_list(gs);
  const unsigned long long* lmass = topk_mass(gs);
  const int tid = threadIdx.x;
  if (tid == 0) gs.bc32[4] = 0xFFFFFFFFu;
  cta_sync();
  if (uint32_t(tid) < len) {
    const uint32_t id = ~uint32_t(list[tid]);
    const uint64_t e = lmass[tid];
    uint64_t run = 0;
    for (uint32_t j = 0; j < len; ++j) run += ~uint32_t(list[j]) < id ? lmass[j] : 0ull;
    if (e > 0 && run <= t && t - run < e) gs.bc32[4] = id;
  }
  cta_sync();
  const uint32_t tok = gs.bc32[4];
  cta_sync();
  return tok == 0xFFFFFFFFu ? -1 : int(tok);
}

// One row by the general path (see the top of this file).  `table` is the
// 2^(j/64) table in shared memory.
template <typename T, typename Xf = NoPrep>
__device__ void general_row(GenShared& gs, const FloatPair* table, const SampleArgs& a, int b,
                            const smp_row_params& prm, const Xf& xf = Xf()) {
  const int tid = threadIdx.x;
  const int V = a.vocab;
  const T* row = reinterpret_cast<const T*>(a.logits) + size_t(b) * V;

  // The maximum (fmaxf skips NaN, which orders with -inf; -0 and +0 share a key).
  float tmax = -INFINITY;
  gen_sweep<T, light_pass_vectors<Xf>()>(row, V, [&](int, float z) { tmax = fmaxf(tmax, z); }, xf);
  const uint32_t thread_key_max = order_key<T>(tmax);
  const uint32_t key_max = uint32_t(block_max_u64(uint64_t(thread_key_max), gs.red64));
  const bool greedy = row_is_greedy(prm);
  int flags = 0;
  if (!key_finite<T>(key_max)) flags |= kRowNonFinite;
  else if (!greedy && !sampling_params_valid(prm)) flags |= kRowBadParams;
  if (flags) {
    if (tid == 0) write_error_row(a, b, flags);
    if (a.full_probs)
      for (int i = tid; i < V; i += kThreads) a.full_probs[size_t(b) * V + i] = __int_as_float(0x7FC00000);
    cta_sync();
    return;
  }
  if (greedy) {   // the lowest id holding the maximum
    uint32_t lo = 0xFFFFFFFFu;
    gen_sweep<T>(row, V, [&](int i, float z) {
      if (order_key<T>(z) == key_max) lo = min(lo, uint32_t(i));
    }, xf);
    const uint32_t argmax = ~uint32_t(block_max_u64(uint64_t(~lo), gs.red64));
    if (tid == 0) {
      a.out_ids[b] = int32_t(argmax);
      if (a.out_probs) a.out_probs[b] = 1.0f;
      if (a.kept) a.kept[b] = 1;
    }
    if (a.full_probs)
      for (int i = tid; i < V; i += kThreads) a.full_probs[size_t(b) * V + i] = uint32_t(i) == argmax ? 1.0f : 0.0f;
    cta_sync();
    return;
  }

  KeptSet ks;
  // vectors in flight in the candidate pass: three binary32 vectors keep the
  // sampler kernel within its registers
  constexpr int kListU = sizeof(T) == 4 ? 3 : kTopU;
  const bool listed = topk_bounded(prm, V) &&
                      gen_kept_set_topk<T, kListU>(row, V, gs, table, prm, key_max, thread_key_max, &ks, xf);
  if (!listed) ks = gen_kept_set<T>(row, V, gs, table, prm, key_max, xf);
  auto mass_of = [&](int i, float z) -> uint64_t { return kept_mass<T>(ks, table, i, z); };
  const uint64_t z_kept = ks.z_kept;
  const uint64_t len = ks.len;
  // The draw: the first kept token (id order) whose running mass exceeds
  // t = floor(u * Z_S), u = Philox draw 0 of row b.
  const uint64_t u53 = uniform53(a.seed, a.offset, a.row_base + uint64_t(b), 0);
  const uint64_t t = uint64_t((u128(u53) * z_kept) >> 53);
  const int tok = listed ? topk_draw(gs, uint32_t(len), t) : gen_walk<T, uint64_t>(row, V, t, gs, mass_of, xf);
  if (tid == 0) {
    a.out_ids[b] = tok;
    if (a.out_probs)
      a.out_probs[b] = tok >= 0 ? float(double(mass_of(tok, xf(tok, Elem<T>::widen(row[tok])))) / double(z_kept))
                                : __int_as_float(0x7FC00000);
    if (a.kept) a.kept[b] = int32_t(len);
  }
  if (a.full_probs) {
    const float zf = float(z_kept);
    for (int i = tid; i < V; i += kThreads) {
      const uint64_t e = mass_of(i, xf(i, Elem<T>::widen(row[i])));
      a.full_probs[size_t(b) * V + i] = e ? __fdiv_rn(float(e), zf) : 0.0f;
    }
  }
  cta_sync();
}
