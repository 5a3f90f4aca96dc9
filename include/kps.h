/*
 * kps.h — C ABI of the GB300 (sm_103a) decode-step token sampler.
 *
 * One call runs the whole per-step sampling post-process over a [B, V]
 * logits matrix, row by row:
 *
 *   1. repetition penalty over the row's seen ids (a CSR list, or with
 *        kps_sample_step a bit set kept on the device across steps)
 *        x = x > 0 ? x / penalty : x * penalty, once per distinct id
 *        (MiniMind "Chapter 10: inference generation", §10.7; the C++
 *        post-processing blog, repetition_penalty section);
 *   2. temperature: x = x / temperature (MiniMind ch.10, §10.4);
 *   3. top-k: keep exactly the first k elements in the order "value
 *        descending, index ascending" when 1 <= k <= min(V, 1024), skip the
 *        stage otherwise (Ascend "torch_npu.npu_top_k_top_p_sample", topK
 *        item 2; MiniMind ch.10, §10.5);
 *   4. top-p: keep the shortest prefix of that order whose softmax mass
 *        reaches top_p (at least one element; top_p <= 0 keeps one element,
 *        top_p >= 1 or NaN skips the stage) (Ascend page, topP full-sort
 *        formula; MiniMind ch.10, §10.6);
 *   5. exponential race: index = argmax over the kept set of
 *        softmax(filtered) / (q + eps), lower index on an exact tie
 *        (Ascend page, "Sample" formulas).
 *
 * It writes the chosen index per row and, when need_logits is set, the
 * filtered logits in vocabulary order: the transformed value at kept
 * positions and -inf elsewhere (Ascend page, logits_top_kp_select).
 *
 * Value conventions (readings where the pages are silent):
 *   - NaN logits are treated as -inf;
 *   - a row whose temperature is not finite and > 0 is greedy: no division,
 *     only the best (penalised) element is kept and chosen;
 *   - a penalty <= 0 or NaN disables the penalty for that row; seen ids
 *     outside [0, V) are ignored; duplicate ids are applied once;
 *   - softmax weights are exp(x - max) with weight 1 at the maximum itself;
 *   - race scores that are NaN are ignored; if every score is NaN the first
 *     element of the order is chosen.
 *
 * Memory: every pointer argument of kps_sample is a DEVICE pointer owned by
 * the caller.  The library allocates nothing, keeps no per-call state and
 * never synchronises the stream.  Calls on different streams are
 * independent provided they use different workspaces and outputs.
 *
 * Errors: argument checks run on the host before anything is launched and
 * return a status code.  A launch failure returns KPS_ERR_CUDA.  Faults the
 * kernel detects itself (a bounded wait that ran out) are recorded in the
 * workspace status word; read them with kps_last_device_status().
 */
#ifndef KPS_H_
#define KPS_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { KPS_F32 = 0, KPS_BF16 = 1 } kps_dtype;

typedef enum {
  KPS_OK = 0,
  KPS_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad dtype, bad eps      */
  KPS_ERR_UNSUPPORTED = 2,  /* V too large for the on-chip row layout          */
  KPS_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small      */
  KPS_ERR_CUDA = 4,         /* a CUDA runtime call or the launch failed        */
  KPS_ERR_TIMEOUT = 5       /* device side: a bounded wait ran out             */
} kps_status;

/* Bytes of device workspace for the fastest schedule of a [B, V] call of
 * dtype dt (256-byte aligned start required).  The first 256 bytes hold the
 * device status word.  For V > 4096 one 32896-byte record per row follows
 * (min(B, 1024) records): the pre-pass of the top-p-only rows merges their
 * bin sums and race words there, and the row kernel reads and clears them.
 * kps_sample accepts any workspace of at least 256 bytes; rows beyond the
 * records it holds run their whole selection inside the row kernel instead.
 * Zero the workspace once before its first use: every call leaves the
 * records zeroed again (the status word aside, which kps_last_device_status
 * reads and clears).  One call at a time may use a workspace.  Returns 0 for
 * invalid sizes. */
size_t kps_workspace_size(int64_t B, int64_t V, kps_dtype dt);

/* Largest vocabulary size kps_sample accepts for dtype dt on the current
 * device (the whole row must fit in the shared memory of one thread-block
 * cluster). */
int64_t kps_max_vocab(kps_dtype dt);

/*
 * kps_sample — the fused sampling step (see the file comment for the math).
 *
 *   logits        [B, V] row-major, fp32 or bf16 (dt), read only.
 *   top_k         [B] int32.  Stage active iff 1 <= top_k[b] <= min(V, 1024).
 *   top_p         [B] fp32.
 *   temperature   [B] fp32.
 *   seen_indptr   [B+1] int32 CSR row pointer into seen_ids, or NULL.
 *   seen_ids      [nnz] int32 token ids already generated per row, or NULL.
 *   penalty       [B] fp32 repetition penalty, or NULL.  The penalty stage
 *                 runs only when all three of seen_indptr, seen_ids and
 *                 penalty are non-NULL.
 *   q             [B, V] fp32 race weights (Exp(1) draws supplied by the
 *                 caller), or NULL to sample off: each row's index is then
 *                 the first element of its kept set's order (the argmax of
 *                 the filtered row, the lowest index among equal maxima;
 *                 the Ascend page's scenario table lets the Sample stage be
 *                 disabled, and the MiniMind inference chapter's greedy mode
 *                 takes that argmax).  The filtered row is the same either
 *                 way.
 *   eps           added to q before dividing; must be >= 0 and finite.
 *   need_logits   non-zero: write out_filtered.
 *   out_idx       [B] int64 chosen token per row.
 *   out_filtered  [B, V] fp32; required iff need_logits.
 *   workspace     device buffer, 256-byte aligned, of at least 256 bytes;
 *                 kps_workspace_size(B, V, dt) bytes for the fastest
 *                 schedule.  Zeroed before its first use (see above).
 *   stream        CUDA stream the work is queued on (0 = legacy default).
 *
 * B == 0 is a valid no-op.  Returns KPS_OK once the work is queued.
 */
kps_status kps_sample(const void* logits, kps_dtype dt, int64_t B, int64_t V,
                      const int32_t* top_k, const float* top_p, const float* temperature,
                      const int32_t* seen_indptr, const int32_t* seen_ids,
                      const float* penalty, const float* q, float eps, int need_logits,
                      int64_t* out_idx, float* out_filtered,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * kps_sample_seeded — kps_sample racing with Exp(1) draws the library generates
 * instead of a caller-supplied q, so no q is read from memory.  The draw of
 * row b, token v is Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel
 * Random Numbers: As Easy as 1, 2, 3", SC'11) with key (seed low 32 bits,
 * seed high 32 bits) on the counter (v / 4, b, step low, step high), output
 * word v mod 4: u = (2 (w >> 9) + 1) 2^-24 and q = -log(u).  Counter-based:
 * any row or token can be drawn alone, and results do not depend on the
 * launch shape.  Change `step` (or `seed`) between decode steps.  Every other
 * argument, result and error is that of kps_sample.
 */
kps_status kps_sample_seeded(const void* logits, kps_dtype dt, int64_t B, int64_t V,
                             const int32_t* top_k, const float* top_p, const float* temperature,
                             const int32_t* seen_indptr, const int32_t* seen_ids,
                             const float* penalty, unsigned long long seed, unsigned long long step,
                             float eps, int need_logits, int64_t* out_idx, float* out_filtered,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * kps_sample_step — one decode step's sampling with every option: the draws
 * (supplied, generated or none), the end-of-sequence epilogue of a
 * generation loop (MiniMind, "Chapter 10: inference generation", the
 * generate loop: a finished sequence emits the end-of-sequence token, a
 * sequence that emits it becomes finished, and the loop stops once all are
 * finished), applied inside the kernel as each row's index is written, and
 * a seen set kept on the device across steps (the same chapter's
 * repetition penalty runs over the distinct ids of the sequence so far, to
 * which each step appends its token: with seen_bits and update_seen the
 * kernel sets that token's bit instead of the caller rebuilding the list).
 */
typedef struct {
  const float* q;            /* [B, V] fp32 draws as for kps_sample, or NULL
                                (sampling off) — ignored when generate != 0 */
  int generate;              /* non-zero: draws generated from (seed, step) as
                                for kps_sample_seeded */
  unsigned long long seed, step;
  unsigned char* finished;   /* [B] device flags, read and updated (0 or 1), or
                                NULL: no epilogue.  A row flagged finished
                                emits eos_id (its filtered row is still
                                written); a row that emits eos_id is flagged. */
  int64_t eos_id;            /* the end-of-sequence token */
  int* unfinished;           /* device int, or NULL: set to the number of rows
                                left unfinished after the step (0: the loop can
                                stop).  Requires finished. */
  uint32_t* seen_bits;       /* [B, (V + 31) / 32] uint32 device, 4-byte aligned,
                                or NULL: the seen set as bits in place of the
                                seen ids (bit v % 32 of word b * ((V + 31) / 32)
                                + v / 32 marks token v of row b; bits of tokens
                                >= V are ignored).  With seen_bits the
                                seen_indptr and seen_ids arguments must be NULL
                                (KPS_ERR_INVALID_ARG otherwise); the penalty runs
                                when penalty is non-NULL, as with the ids. */
  int update_seen;           /* non-zero: after the step each row's emitted token
                                (the index written to out_idx, after the
                                end-of-sequence epilogue) joins its seen set, the
                                one bit set in place — the generate loop's
                                appended token, so the next step needs no new
                                seen list.  Requires seen_bits. */
  int kernel_policy;         /* which kernel runs this call (for tests and tuning;
                                both compute the same results):
                                0 = automatic (kps_sample and kps_sample_seeded
                                    always use it): the row kernel — one CTA per
                                    row (both CTAs of a 2-CTA cluster per row when
                                    the batch gives every row a cluster of its
                                    own), the row read from global memory with
                                    16-byte loads, two CTAs per SM — for batches
                                    of at least 64 rows whose rows are 16-byte
                                    aligned and V <= 262144; the cluster kernel —
                                    one thread-block cluster per row, the row
                                    resident in the cluster's shared memory —
                                    otherwise;
                                1 = always the cluster kernel;
                                2 = the row kernel whenever the shape allows it;
                                3 = as 2, with the row kernel's exact whole-row
                                    selection forced on every row (the path it
                                    takes when its sample misses); slow.
                                Other values: KPS_ERR_INVALID_ARG.  The library
                                keeps no kernel choice between calls. */
} kps_step_opts;

kps_status kps_sample_step(const void* logits, kps_dtype dt, int64_t B, int64_t V,
                           const int32_t* top_k, const float* top_p, const float* temperature,
                           const int32_t* seen_indptr, const int32_t* seen_ids,
                           const float* penalty, const kps_step_opts* opts, float eps,
                           int need_logits, int64_t* out_idx, float* out_filtered,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Reads (and clears) the device status word of a workspace: waits for the
 * stream, stores KPS_OK or the first device-side error code in *out. */
kps_status kps_last_device_status(void* workspace, cudaStream_t stream, int* out);

/*
 * kps_sample_noalloc — kps_sample for callers that cannot allocate device
 * memory.  Some hosts of this library cannot call cudaMalloc: an allocator
 * that owns all device memory and forbids outside allocations, a real-time
 * path where allocation latency or failure is not acceptable, or code that
 * runs under a memory budget it does not control.  This entry point needs no
 * workspace: its scratch (a 256-byte workspace: the device status word)
 * lives in a fixed array inside the library, 4096 bytes, held on every GPU
 * that loads the library until the process exits.  It therefore never runs
 * the pre-pass of the top-p-only rows.  It allocates nothing and calls no allocating
 * routine; the caller still passes inputs and outputs as for kps_sample.
 * (The method's pages have no counterpart to this entry point.)
 *
 *   - Arguments, results and math are exactly those of kps_sample.
 *   - The first call on each device looks up the scratch array's device
 *     address with that device current (and sets kernel attributes); make
 *     that first call before capturing the stream into a CUDA graph.
 *   - Every call on a device shares the one scratch array, which keeps the
 *     last call's contents; each call clears it on its stream first.  Calls
 *     that overlap on the GPU (different streams, no ordering between them)
 *     race on it.  A device-side timeout is recorded there but cannot be read
 *     back through this entry point.
 */
kps_status kps_sample_noalloc(const void* logits, kps_dtype dt, int64_t B, int64_t V,
                              const int32_t* top_k, const float* top_p, const float* temperature,
                              const int32_t* seen_indptr, const int32_t* seen_ids,
                              const float* penalty, const float* q, float eps, int need_logits,
                              int64_t* out_idx, float* out_filtered, cudaStream_t stream);


/* Which kernel the most recent kps_sample call of the calling host thread
 * that launched one used: 1 = the cluster kernel (kps_sample_kernel),
 * 2 = the row kernel (kps_row_kernel, possibly after its pre-pass
 * kps_prepass_kernel), 0 = none yet. */
int kps_last_kernel(void);

/* Kernels the most recent kps_sample call of the calling host thread that
 * launched any queued: 1, or 2 when the row kernel was preceded by its
 * pre-pass over the top-p-only rows (kps_prepass_kernel); 0 = none yet. */
int kps_last_launch_count(void);

/* CTAs per thread-block cluster of the kernel that the most recent kps_sample
 * call of the calling host thread launched (for the cluster kernel: the CTAs
 * that share one row); 0 = none yet.  Matches the cluster_size that
 * kps_query_launch reports for the same (B, V, dt) under the automatic policy
 * whenever that call took the cluster kernel. */
int kps_last_cluster_size(void);

/* Static description of a status code. */
const char* kps_status_string(kps_status s);

/* Launch shape kps_sample would use for (B, V, dt) on the current device:
 * cluster size (CTAs per row), elements per CTA, dynamic shared memory per
 * CTA in bytes.  Returns KPS_OK or an error for unsupported sizes. */
kps_status kps_query_launch(int64_t B, int64_t V, kps_dtype dt, int* cluster_size,
                            int64_t* chunk_elems, size_t* smem_bytes);

#ifdef __cplusplus
}
#endif

#endif /* KPS_H_ */
