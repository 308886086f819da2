/*
 * smp.h -- C ABI of libsmp: a batched next-token sampler and a
 * speculative-decoding verifier for NVIDIA GB300 (sm_103a).
 *
 * Every entry point is asynchronous on the caller's CUDA stream, allocates
 * nothing, and reads and writes only the caller-owned device buffers it is
 * given (smp_spec_verify_static also its own fixed scratch array).  Host-detectable errors (a NULL pointer, a size out of range, an
 * unknown dtype) return a status code before anything is launched.  Problems
 * that belong to one row (bad knobs, no finite logit, a draft id out of range,
 * a wait that ran out of time) give that row the id -1 and OR a flag
 * (SMP_ROW_*) into the optional device status word, which the call clears
 * first.
 *
 * Random numbers: every draw uses Philox4x64-10 (Salmon et al., "Parallel
 * Random Numbers: As Easy as 1, 2, 3", SC'11) with key (seed, 0) and counter
 * (offset, row, draw, 0); the uniform is the top 53 bits of the first output
 * word.  The same (seed, offset) reproduces a call bit for bit, whatever the
 * launch shape.
 *
 * Probability masses: the device represents exp((z - max z) / T) of every
 * token as a 64-bit fixed-point integer E = round(e * 2^44), computed with a
 * double-float exponential (relative error below 2^-44), and sums them
 * exactly in integers.  Masses below 2^-45 of the row maximum (more than
 * about 31 T below the top logit) are zero.
 *
 * Sharding: rows are independent, so a batch split across GPUs (or across
 * calls) gives the same tokens as one call when each part passes the global
 * index of its first row as row_base (smp_sample_rows, smp_spec_verify_rows):
 * the Philox counter holds row_base + row.  The other entry points use
 * row_base = 0.
 *
 * Two departures from the first sketch of this interface, kept on purpose:
 *   - the verifier takes a caller-owned workspace (smp_spec_verify_workspace_bytes):
 *     its per-position statistics are written by one kernel and read by the
 *     next, which shared memory cannot carry between launches; callers that
 *     cannot allocate use smp_spec_verify_static;
 *   - status codes 4 and 5 are SMP_ERR_UNSUPPORTED (a vocabulary beyond
 *     SMP_MAX_VOCAB) and SMP_ERR_WORKSPACE (a missing or short workspace),
 *     host-side conditions of this interface; the device conditions the sketch
 *     gave codes to (a wait that ran out of time, a bad row) are reported per
 *     row through the SMP_ROW_* flags of the status word instead, since they
 *     are only known after the call has returned.
 */
#ifndef SMP_H
#define SMP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SMP_ABI_VERSION 3

/* Largest vocabulary the kernels accept (rows are kept in on-chip memory). */
#define SMP_MAX_VOCAB (1 << 19)
/* Largest number of draft tokens per verify row. */
#define SMP_MAX_DRAFT 16
/* Longest window of recent tokens the repetition penalty looks at. */
#define SMP_MAX_HISTORY 64
/* Most beams per group, and most candidates kept per group, of a beam step. */
#define SMP_MAX_BEAM_WIDTH 32

typedef enum smp_dtype {
    SMP_F32 = 0,   /* IEEE binary32 logits */
    SMP_BF16 = 1   /* bfloat16 logits (upper half of binary32) */
} smp_dtype;

/*
 * Per-row sampling knobs, 20 bytes, little endian, laid out as written.
 *   temperature  T: logits are divided by T before the softmax ("Decoding &
 *                Speculative Sampling", section 39.2).  T == 0 means greedy;
 *                T < 0, NaN or infinite makes the row invalid.
 *   top_k        keep the k most likely tokens (ties: lower id first), active
 *                for 0 < top_k < V; top_k < 0 is invalid.
 *   top_p        keep the shortest most-likely prefix whose probability
 *                reaches top_p (at least one token); off for top_p >= 1;
 *                top_p < 0 or NaN is invalid.
 *   min_p        keep p_i >= min_p * max_j p_j ("Inference: Sampling, the KV
 *                Cache, Speculative Decoding and int8", section "Picking the
 *                next token"); active for 0 < min_p < 1 only, which is the
 *                range in which that section's own code applies the filter:
 *                0 and every value >= 1 switch it off (so min_p = 1 does not
 *                keep just the tied arg-max set); min_p < 0 or NaN is invalid.
 *   greedy       non-zero: take the arg-max (lowest id on ties), knobs ignored.
 * The filters are applied to the same post-temperature distribution and their
 * kept sets intersected, then renormalised (eq. 39.2).
 */
typedef struct smp_row_params {
    float temperature;
    int32_t top_k;
    float top_p;
    float min_p;
    int32_t greedy;
} smp_row_params;

typedef enum smp_status {
    SMP_OK = 0,
    SMP_ERR_INVALID_ARG = 1,   /* NULL pointer, size or count out of range, misaligned base */
    SMP_ERR_DTYPE = 2,         /* dtype is not SMP_F32 or SMP_BF16 */
    SMP_ERR_CUDA = 3,          /* a CUDA runtime call failed (see smp_last_cuda_error) */
    SMP_ERR_UNSUPPORTED = 4,   /* vocabulary too large for the on-chip row layout */
    SMP_ERR_WORKSPACE = 5      /* workspace NULL or smaller than required */
} smp_status;

/* Flags OR-ed into the device status word, one or more per affected row. */
#define SMP_ROW_BAD_PARAMS 1   /* invalid knobs on a sampling or verify row */
#define SMP_ROW_NONFINITE 2    /* the row's maximum logit is not finite (all -inf/NaN, or +inf) */
#define SMP_ROW_TIMEOUT 4      /* a bounded wait between the CTAs of a row ran out of time */
#define SMP_ROW_BAD_DRAFT 8    /* a draft id outside [0, V) */

/*
 * smp_sample -- draw one token per row from temperature / top-k / top-p /
 * min-p filtered, renormalised distributions ("Decoding & Speculative
 * Sampling", section 39.2 and eq. 39.2; the draw walks the kept tokens in id
 * order and stops where the running total passes u: "Choosing the next word",
 * section "Where the randomness comes from, and where it stops").
 *
 *   logits     device, [batch, vocab] row-major contiguous, dtype elements;
 *              base aligned to the element size.  NaN counts as -inf.
 *   batch      rows, 1 .. 2^31-1;  vocab: 1 .. SMP_MAX_VOCAB.
 *   params     device, [batch] smp_row_params.
 *   seed, offset  Philox key and per-step counter; row b uses draw 0.
 *   out_ids    device, [batch] int32: the token, or -1 for an error row.
 *   out_probs  device, [batch] float or NULL: p~ of the token (1 for greedy,
 *              NaN for an error row).
 *   status     device, one int32 or NULL: cleared, then OR of SMP_ROW_* flags.
 *   stream     a cudaStream_t (NULL: the legacy default stream).
 * Returns SMP_OK once the work is queued.
 */
smp_status smp_sample(const void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                      const smp_row_params* params, uint64_t seed, uint64_t offset,
                      int32_t* out_ids, float* out_probs, int32_t* status, void* stream);

/*
 * smp_filter_debug -- as smp_sample, and also writes the renormalised
 * distribution p~ of eq. 39.2 of every row and the size of its kept set.
 *   out_probs_full  device, [batch, vocab] float: p~_i (0 outside the kept
 *                   set; one-hot for greedy rows; NaN for error rows).
 *   out_kept        device, [batch] int32: |S| (1 for greedy, 0 for errors).
 * Meant for tests; it moves 4 bytes per logit more than smp_sample.
 */
smp_status smp_filter_debug(const void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                            const smp_row_params* params, uint64_t seed, uint64_t offset,
                            int32_t* out_ids, float* out_probs, float* out_probs_full,
                            int32_t* out_kept, int32_t* status, void* stream);

/*
 * smp_sample_processed -- smp_sample after a logit pre-pass: a repetition
 * penalty over recent tokens and a constraint mask.
 *
 *   repetition penalty  for each distinct token id i among the row's recent
 *                tokens, z_i <- z_i / r if z_i > 0, else z_i * r ("Choosing
 *                the next word", section "The repetition penalty"), applied
 *                to the raw logits; the result is computed in binary32 and
 *                kept in the logits' precision (bf16 logits: rounded to the
 *                nearest bf16, ties to even).
 *   constraint mask  tokens outside the allowed set get the logit -inf, so
 *                the distribution is the model's conditioned on the allowed
 *                set ("Decoding & Speculative Sampling", section 39.3).
 * Then temperature, filters and the draw run exactly as in smp_sample.
 *
 *   allowed      device, [batch, ceil(vocab / 32)] uint32, or NULL (no mask):
 *                bit (i mod 32) of word i / 32 set when token i is allowed.
 *                A row with no allowed token has no finite logit: id -1 and
 *                SMP_ROW_NONFINITE.
 *   history      device, [batch, history_len] int32 recent token ids, or NULL;
 *                ids outside [0, vocab) are padding, repeated ids count once.
 *   history_len  0 .. SMP_MAX_HISTORY.
 *   repetition_penalty  device, [batch] float r, or NULL (no penalty); r = 1
 *                leaves the row unchanged; r must be finite and > 0, else the
 *                row is an error row (SMP_ROW_BAD_PARAMS, greedy or not).
 * Every other argument and the error behaviour are those of smp_sample.
 * The pre-pass runs inside smp_sample's own single pass over the logits
 * (each value is transformed as it is read), so the cost over smp_sample is
 * the mask words (vocab / 8 bytes per row) and the transform of the units
 * that hold a disallowed token or a history id.
 */
smp_status smp_sample_processed(const void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                                const smp_row_params* params, const uint32_t* allowed, const int32_t* history,
                                int32_t history_len, const float* repetition_penalty, uint64_t seed,
                                uint64_t offset, int32_t* out_ids, float* out_probs, int32_t* status,
                                void* stream);

/*
 * smp_sample_rows -- smp_sample_processed for a part of a larger batch: the
 * Philox counter of row b is row_base + b, so splitting a batch into parts
 * (over GPUs or calls) and passing each part's first global row index gives
 * exactly the tokens of one call on the whole batch.  allowed, history and
 * repetition_penalty may all be NULL (no pre-pass: the call is smp_sample
 * with a row base).  Every other argument and the error behaviour are those
 * of smp_sample_processed.
 */
smp_status smp_sample_rows(const void* logits, int32_t batch, int32_t vocab, smp_dtype dtype,
                           const smp_row_params* params, const uint32_t* allowed, const int32_t* history,
                           int32_t history_len, const float* repetition_penalty, uint64_t seed, uint64_t offset,
                           uint64_t row_base, int32_t* out_ids, float* out_probs, int32_t* status, void* stream);

/*
 * smp_logit_prepass -- the pre-pass of smp_sample_processed written into the
 * logits in place, so that smp_sample, or a verifier call, then reads the
 * processed logits.  For callers whose later steps all need the processed
 * logits (the verifier has no pre-pass of its own); to sample once,
 * smp_sample_processed is faster.
 *
 *   logits       device, [batch, vocab] contiguous, dtype elements, read and
 *                written: disallowed tokens become -inf, each distinct
 *                allowed history id gets z / r (z > 0) or z * r (z <= 0),
 *                computed in binary32 and stored in the logits' precision
 *                (bf16: nearest, ties to even).  Nothing else is written.
 *   allowed, history, history_len, repetition_penalty  as for
 *                smp_sample_processed.
 *   status       device int32 or NULL: cleared, then SMP_ROW_BAD_PARAMS for
 *                rows whose factor r is not finite and > 0.  Such rows are
 *                filled with NaN, so that a following smp_sample gives them
 *                id -1 and SMP_ROW_NONFINITE.
 * Cost: the mask words are read (vocab / 8 bytes per row) and only changed
 * elements are written; a row without a mask and without a penalty is not
 * touched.
 */
smp_status smp_logit_prepass(void* logits, int32_t batch, int32_t vocab, smp_dtype dtype, const uint32_t* allowed,
                             const int32_t* history, int32_t history_len, const float* repetition_penalty,
                             int32_t* status, void* stream);

/*
 * smp_spec_verify_workspace_bytes -- device workspace smp_spec_verify needs
 * for a batch of `batch` rows with `k` drafts (0 if the sizes are invalid).
 */
size_t smp_spec_verify_workspace_bytes(int32_t batch, int32_t k);

/*
 * smp_spec_verify -- speculative-decoding verification of a batch ("Decoding
 * & Speculative Sampling", section 39.4, eqs. 39.3 and 39.4; "Speculative
 * decoding -- Hinglish notes", section "The Algorithm (Step-by-Step)").
 * For each row b and i = 0..K-1 in order, draft x = draft_ids[b, i] is kept
 * when u_i < p_i(x) / max(q_i(x), 1e-300) with p_i = softmax(p_logits[b, i]),
 * q_i = softmax(q_logits[b, i]) (temperature 1, no filters).  At the first
 * rejection j the replacement is drawn from max(0, p_j - q_j) renormalised
 * (from p_j if that mass is zero); if all K are kept a bonus token is drawn
 * from softmax(p_logits[b, K]).  u_i is draw i of row b; the replacement or
 * bonus uses draw K.
 *
 *   p_logits   device, [batch, k+1, vocab] contiguous, dtype elements.
 *   q_logits   device, [batch, k, vocab] contiguous, same dtype.
 *   draft_ids  device, [batch, k] int32.
 *   batch 1 .. 2^20;  k 1 .. SMP_MAX_DRAFT;  vocab 1 .. SMP_MAX_VOCAB.
 *   out_accepted_len  device, [batch] int32: accepted drafts 0..k (-1: error).
 *   out_ids    device, [batch, k+1] int32: the accepted drafts, then the
 *              replacement or bonus token, then -1 padding.
 *   status     device int32 or NULL, as for smp_sample.
 *   workspace  device buffer of at least smp_spec_verify_workspace_bytes(batch, k)
 *              bytes, 8-byte aligned; owned by the caller, contents scratch.
 *              Calls that overlap on the GPU must not share it.
 */
smp_status smp_spec_verify(const void* p_logits, const void* q_logits, const int32_t* draft_ids,
                           int32_t batch, int32_t k, int32_t vocab, smp_dtype dtype,
                           uint64_t seed, uint64_t offset, int32_t* out_accepted_len,
                           int32_t* out_ids, int32_t* status, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * smp_spec_verify_params -- smp_spec_verify with per-row knobs: temperature
 * and filters on both distributions, or greedy verification.
 *
 *   temperature  p_T = softmax(p_logits / T) and q_T = softmax(q_logits / T)
 *                replace p and q everywhere above; the accept rule
 *                min(1, p_T(x) / q_T(x)) is unchanged ("Speculative decoding
 *                -- Hinglish notes", section "Temperature and Sampling").
 *   top_k, top_p, min_p  the filters that are on (as in smp_sample) apply to
 *                every target and draft row: p and q become the renormalised
 *                filtered distributions p~ and q~ of eq. 39.2 ("Decoding &
 *                Speculative Sampling", section 39.2), selected exactly as
 *                the sampler selects them, and the accept, residual and bonus
 *                rules run on p~ and q~, so the output follows the target's
 *                filtered distribution.  A draft outside the draft's kept
 *                set has q~(x) = 0 (kept iff p~(x) > 0); one outside the
 *                target's kept set is rejected.  Filtered rows take an exact
 *                selection per logit row (several passes over it), so they
 *                cost more than unfiltered ones.
 *   greedy       (the flag, or T == 0) a draft is kept when it is the
 *                target's arg-max at its position (lowest id on ties); at the
 *                first mismatch j the target's arg-max of position j is
 *                emitted, and if all K are kept the arg-max of position K.
 *                The output is then exactly greedy decoding with the target
 *                ("Inference: Sampling, the KV Cache, Speculative Decoding
 *                and int8", section "Speculative decoding").  No uniform is
 *                used and q_logits is not read for that row (its values,
 *                finite or not, do not matter); the other knobs are ignored.
 *   params       device, [batch] smp_row_params, or NULL for T = 1 and no
 *                filters on every row (then, without out_alpha, the call is
 *                smp_spec_verify).  Knob validity is the sampler's; a row
 *                with invalid knobs gets accepted length -1, ids -1 and
 *                SMP_ROW_BAD_PARAMS.
 *   out_alpha    device, [batch, k] float, or NULL: the acceptance rate of
 *                every draft position, alpha_i = sum_x min(p_i(x), q_i(x))
 *                on the compared distributions (after temperature and
 *                filters), the probability that a proposal drawn from q_i
 *                is kept ("Decoding & Speculative Sampling", section 39.4
 *                and Listing 39.5), computed for all k positions whatever
 *                was accepted; within about 1e-5 (binary32 probabilities,
 *                exact fixed-point sums).  NaN for greedy rows (no q is
 *                compared) and error rows.  It costs one more pass over the
 *                k (p, q) row pairs, normally from L2.
 * Every other argument, the workspace and the error behaviour are those of
 * smp_spec_verify.
 */
smp_status smp_spec_verify_params(const void* p_logits, const void* q_logits, const int32_t* draft_ids,
                                  int32_t batch, int32_t k, int32_t vocab, smp_dtype dtype,
                                  const smp_row_params* params, uint64_t seed, uint64_t offset,
                                  int32_t* out_accepted_len, int32_t* out_ids, float* out_alpha,
                                  int32_t* status, void* workspace, size_t workspace_bytes, void* stream);

/*
 * smp_spec_verify_rows -- smp_spec_verify_params for a part of a larger batch:
 * the uniforms of batch row b are drawn at Philox counter row row_base + b
 * (draws 0..k), so parts verified separately with their first global row
 * index give exactly the result of one call on the whole batch.  Every other
 * argument, the workspace and the error behaviour are those of
 * smp_spec_verify_params.
 */
smp_status smp_spec_verify_rows(const void* p_logits, const void* q_logits, const int32_t* draft_ids,
                                int32_t batch, int32_t k, int32_t vocab, smp_dtype dtype,
                                const smp_row_params* params, uint64_t seed, uint64_t offset, uint64_t row_base,
                                int32_t* out_accepted_len, int32_t* out_ids, float* out_alpha, int32_t* status,
                                void* workspace, size_t workspace_bytes, void* stream);

/*
 * smp_beam_topk_workspace_bytes -- device workspace smp_beam_topk needs (0 if
 * the sizes are invalid).
 */
size_t smp_beam_topk_workspace_bytes(int32_t groups, int32_t beams, int32_t width);

/*
 * smp_beam_topk -- the candidate selection of one beam-search step ("Decoding
 * & Speculative Sampling", section 39.1, eq. 39.1 and Listing 39.1;
 * "Efficient Inference & Compression", section "Beam search").  For each
 * group (one request), every beam b is extended by every token t with score
 * s_b + log p_b(t), p_b = softmax(logits[g, b]) (temperature 1, no filters),
 * and the `width` best candidates of the group's beams x vocab are returned,
 * best first; equal scores keep the lower flat index b * vocab + t first (the
 * listing's stable sort).
 *
 *   logits       device, [groups, beams, vocab] contiguous, dtype elements.
 *   beam_scores  device, [groups, beams] double: s_b (log-probabilities of the
 *                prefixes); -inf marks a dead beam, NaN makes an error group.
 *   groups 1 ..; beams, width 1 .. SMP_MAX_BEAM_WIDTH; vocab 1 .. SMP_MAX_VOCAB.
 *   out_parent, out_token  device, [groups, width] int32: the beam each kept
 *                candidate extends and its token; out_score [groups, width]
 *                double: its score.  Ranks past beams x vocab, and every rank
 *                of an error group, are -1 / NaN.
 *   status       device int32 or NULL: SMP_ROW_NONFINITE (a beam with no
 *                finite logit), SMP_ROW_BAD_PARAMS (a NaN beam score).
 *   workspace    device buffer of smp_beam_topk_workspace_bytes(groups,
 *                beams, width) bytes, 8-byte aligned; caller-owned scratch.
 * log p is computed as z - m - ln Z with Z a sum of binary32 exponentials in
 * fixed point (relative error below about 1e-6), so scores match an fp64
 * log-softmax within about 1e-6; candidates closer than that may swap.
 */
smp_status smp_beam_topk(const void* logits, const double* beam_scores, int32_t groups, int32_t beams,
                         int32_t vocab, int32_t width, smp_dtype dtype, int32_t* out_parent, int32_t* out_token,
                         double* out_score, int32_t* status, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * Size of the device array that smp_spec_verify_static uses as its workspace
 * (1 MiB: enough for batch * (2k+1) <= 32768, e.g. 1024 rows with k = 15).
 */
#define SMP_STATIC_VERIFY_SCRATCH_BYTES (1u << 20)

/*
 * smp_spec_verify_static -- smp_spec_verify for callers that cannot allocate
 * device memory.  The pages have no counterpart to this call; it exists for
 * the deployment, not for the method.
 *
 * Some callers cannot hand the verifier a workspace: code that runs inside an
 * allocator or memory-pool callback, runtimes that forbid cudaMalloc once they
 * have started serving, or loops that must not let cudaMalloc / cudaFree
 * synchronise the device.  This entry point takes the same arguments as
 * smp_spec_verify minus the workspace, and allocates nothing: its scratch is
 * a fixed array of SMP_STATIC_VERIFY_SCRATCH_BYTES in device memory that the
 * library holds on every GPU that loads it, until the process exits.
 *
 *   - Sizes whose workspace (smp_spec_verify_workspace_bytes(batch, k)) is
 *     larger than SMP_STATIC_VERIFY_SCRATCH_BYTES return SMP_ERR_WORKSPACE
 *     before anything is launched.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture on the device.  The address is kept for the
 *     rest of the process, which assumes one CUDA context per device (the
 *     primary context) for the process lifetime: after cudaDeviceReset, or
 *     with another context made current on that device, the kept address no
 *     longer names the array and this entry point must not be called.
 *   - Every call on a device uses the same array and leaves its contents
 *     behind.  Each call writes every entry it reads before reading it, so
 *     nothing needs to start at zero, but calls that can overlap on the GPU
 *     (different streams without ordering between them) race on the array and
 *     must not be issued.
 */
smp_status smp_spec_verify_static(const void* p_logits, const void* q_logits, const int32_t* draft_ids,
                                  int32_t batch, int32_t k, int32_t vocab, smp_dtype dtype,
                                  uint64_t seed, uint64_t offset, int32_t* out_accepted_len,
                                  int32_t* out_ids, int32_t* status, void* stream);

/* Human-readable name of a status code (static string). */
const char* smp_status_string(smp_status s);

/* cudaError_t value of the last SMP_ERR_CUDA returned on this thread. */
int32_t smp_last_cuda_error(void);

/* SMP_ABI_VERSION of the loaded library. */
int32_t smp_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SMP_H */
