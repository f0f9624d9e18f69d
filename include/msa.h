/*
 * msa.h - C ABI of libmsa: block-sparse, causal, document-local grouped-query
 * attention (MiniMax Sparse Attention, "MSA") forward and backward on one
 * NVIDIA GB300 (sm_103a).
 *
 * What the library computes is fixed by the flat-attention interface of the
 * NeMo-Automodel PR "feat(minimax-m3): add SM100 MSA sparse attention with
 * custom backward" (sections "Design" and "Supported scope") and by the
 * run_backward contract on the API page "msa_backward_sm100":
 *
 *   Q, dO : bf16 [T, 64, 128]   compact token-major (THD) rows
 *   K, V  : bf16 [T, 4, 128]
 *   q2k   : int32 [4, T, 16]    document-local key-block ids per index head,
 *                               -1 marks an unused slot
 *   doc_offsets : int32 [D+1]   0 = o_0 < o_1 < ... < o_D = T
 *
 * Query head h reads KV head and index head g = h / 16.  Token t = o_d + p of
 * document d attends key o_d + j iff j <= p and floor(j / 128) is one of the
 * values in q2k[g, t, :] (a set: duplicates count once).  Then
 *   s_j = scale * <Q[t,h], K[j,g]>,  LSE[t,h] = ln sum_j exp(s_j),
 *   O[t,h] = sum_j exp(s_j - LSE[t,h]) V[j,g],
 * and the backward returns dQ, dK, dV of L = sum(O * dO).  A row that sees no
 * key gets O = 0, LSE = -inf and zero gradients.  A q2k value < -1 or >= the
 * document's block count is an error (MSA_ERR_BAD_Q2K, detected on device).
 *
 * Conventions for every call:
 *   - All tensor and workspace pointers are DEVICE pointers on the current
 *     CUDA device, contiguous, 16-byte aligned.  The caller owns all memory;
 *     the library never allocates or frees device memory.
 *   - Calls are asynchronous on the given stream (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronise, except the diagnostics
 *     msa_read_status and msa_plan_export which say so.
 *   - Host-detectable problems (null pointer, bad size, misalignment, small
 *     workspace) return an error before anything is launched.  Problems only
 *     the device can see (bad q2k value, bad document offsets, a pipeline
 *     wait that timed out) set bits of the plan's device status word; later
 *     kernels of the same plan then skip their work.  msa_read_status reads it.
 *   - Gradients are accumulated with floating-point atomics, so results are
 *     not bitwise reproducible from run to run.  There is no deterministic
 *     mode.
 *   - Limits: 1 <= T <= 2^20, 1 <= num_docs <= T.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Stream handle: a cudaStream_t, passed as an opaque pointer. */
typedef struct CUstream_st* msa_stream_t;

typedef enum msa_status {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,  /* null pointer, T or num_docs out of range, ...  */
  MSA_ERR_UNSUPPORTED = 2,  /* device is not sm_100 / sm_103 class             */
  MSA_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned                */
  MSA_ERR_WORKSPACE = 4,    /* workspace smaller than the *_workspace_bytes   */
  MSA_ERR_CUDA = 5,         /* a CUDA runtime call failed                      */
  MSA_ERR_BAD_Q2K = 6,      /* device: a q2k slot outside [-1, blocks of doc)  */
  MSA_ERR_BAD_OFFSETS = 7,  /* device: doc_offsets not 0 < ... strictly up .. T */
  MSA_ERR_TIMEOUT = 8,      /* device: a bounded pipeline wait gave up         */
  MSA_ERR_CAPACITY = 9,     /* device: a plan table exceeded its capacity      */
  MSA_ERR_RANGE = 10        /* device warning: the last backward's 16-bit dQ
                               pool overflowed (dQ holds inf / nan); rerun it
                               with MSA_DQ_ACCUM_BF16 or MSA_DQ_ACCUM_F32      */
} msa_status;

/* Human-readable name of a status code (static string). */
const char* msa_status_string(msa_status s);

/* Precision of the dQ accumulation pool of msa_backward.  The pages' default
 * is packed FP16 atomics with a BF16 switch for range (section "Supported
 * scope", the MSA_M3_DQ_ACCUM setting); FP32 is the widest and slowest.
 * FP16 saturates above 65504: when the finalize reads a non-finite FP16 pool
 * value it sets MSA_ERR_RANGE in the plan's status word.  That bit is a
 * warning about the last backward only (every backward clears it first) and,
 * unlike the errors, does not make later kernels of the plan skip work. */
typedef enum msa_dq_accum {
  MSA_DQ_ACCUM_F16 = 0,
  MSA_DQ_ACCUM_BF16 = 1,
  MSA_DQ_ACCUM_F32 = 2
} msa_dq_accum;

/* Precision of the forward's O accumulation pool.  The up-to-16 block
 * partials of an output row are added in a pool at a shared row shift; FP32
 * keeps O's rounding to that of the final bf16 store.  MSA_O_ACCUM_BF16 is
 * rejected with MSA_ERR_UNSUPPORTED: an 8-bit mantissa in every addition
 * plus the bf16 store can put O one bf16 ulp (1.6e-2 at |O| in [2, 4)) off
 * the exact result, above the forward's 1e-2 max-abs bar. */
typedef enum msa_o_accum {
  MSA_O_ACCUM_F32 = 0,
  MSA_O_ACCUM_BF16 = 1
} msa_o_accum;

/* Plan-build options.  Pass NULL for the defaults. */
typedef struct msa_plan_options {
  /* Tasks of one (index head, key block) bucket are cut at runs of
   * super_block consecutive query blocks (0 = never cut).  Default 64. */
  int32_t super_block;
  /* An msa_dq_accum value.  Default MSA_DQ_ACCUM_F16. */
  int32_t dq_accum;
  /* An msa_o_accum value; only (0) MSA_O_ACCUM_F32 is accepted. */
  int32_t o_accum;
  /* Dense octets of the forward: an aligned run of 8 tokens in query block
   * b whose tokens see different blocks runs as one tile over all blocks
   * 0 .. b, each token's rows masked to its own blocks, when b + 1 <=
   * dense_blocks (instead of through the pooled tasks).  0 selects the
   * default, 32; -1 turns dense octets off; 1 .. 64 set the bound; other
   * values give MSA_ERR_INVALID_ARG. */
  int32_t dense_blocks;
  int32_t reserved[4];
} msa_plan_options;

/*
 * The execution plan derived from q2k and the document layout: per index
 * head and key block, the queries that selected it (the k2q CSR), and the
 * task table of 128-row tiles (8 queries x 16 heads of one index head against
 * one key block) that the forward and backward kernels walk.  The pages call
 * these the CSR and scheduling metadata and, on the API page
 * msa_backward_sm100, the backward's task rows, one 128-row tile each,
 * grouped by (batch, index head, key block).
 *
 * A plain struct of device pointers into the caller's plan workspace and of
 * host-side capacities.  Fill it with msa_build_plan; do not edit it.  It
 * stays valid while the workspace and the q2k / doc_offsets buffers live and
 * may be reused by any number of msa_forward / msa_backward calls on the same
 * T, q2k and documents.  All counts live on the device.
 */
typedef struct msa_plan {
  int64_t T;
  int32_t num_docs;
  int32_t super_block;
  int32_t dq_accum;
  int32_t o_accum;
  int32_t dense_blocks; /* the bound in effect (0: no dense octets)     */
  int64_t nb_cap;     /* bound on the number of 128-key blocks            */
  int64_t tri_cap;    /* bound on (index head, doc, key block, query block) */
  int64_t nnz_cap;    /* bound on CSR entries                              */
  int64_t task_cap;   /* bound on tasks                                    */
  const int32_t* q2k;
  const int32_t* doc_offsets;
  int64_t* header;    /* device: status and counts                         */
  int32_t* doc_info;  /* device: [num_docs][4] start, length, blocks, block base */
  int64_t* doc_tri;   /* device: [num_docs+1] prefix of per-doc count entries */
  int32_t* cnt;       /* device: [tri_cap] queries per count entry          */
  int32_t* off;       /* device: [tri_cap] exclusive prefix of cnt          */
  int32_t* col;       /* device: [nnz_cap] query tokens, sorted per entry   */
  int32_t* tcnt;      /* device: [tri_cap] tasks per count entry            */
  int32_t* toff;      /* device: [tri_cap] exclusive prefix of tcnt         */
  int32_t* tasks;     /* device: [task_cap][4] task records                 */
  int32_t* scan_tmp;  /* device: scan scratch                               */
  int64_t scan_tmp_len;
  /* The forward's octet groups: aligned runs of 8 tokens (document positions
   * 8k .. 8k+7, one block b) whose tokens all see the same selected blocks,
   * or whose block range 0 .. b is short (dense octets, each token masked to
   * its own blocks); their tiles are accumulated block after block in one
   * place, without the pool. */
  int64_t item_cap;   /* bound on octet-group items                        */
  uint8_t* grouped;   /* device: [4][T] 1 = the token's octet is grouped    */
  int32_t* items;     /* device: [item_cap][36] group items (msa_plan_export_groups) */
  int32_t* fflag;     /* device: [task_cap] task has an ungrouped query      */
  int32_t* fpos;      /* device: [task_cap] exclusive prefix of fflag        */
  int32_t* ftasks;    /* device: [task_cap][4] the forward's pooled tasks    */
  int32_t* rows;      /* device: [4 T] the (token t, index head g) pairs
                       * outside the octet groups, as 4 t + g, in no
                       * particular order (the pooled path's rows)           */
} msa_plan;

/* Bytes of plan workspace needed for T tokens in num_docs documents.
 * Host only, no CUDA call. */
msa_status msa_plan_workspace_bytes(int64_t T, int32_t num_docs, size_t* bytes);

/*
 * Build the plan on the device (no host synchronisation): validate the
 * document offsets and q2k, invert q2k into the k2q CSR (queries ascending
 * within each bucket), cut the buckets into tasks and count the attended
 * (query, head, key) triples.
 *   q2k          device int32 [4, T, 16]
 *   doc_offsets  device int32 [num_docs + 1]
 *   workspace    device, >= msa_plan_workspace_bytes(T, num_docs)
 *   out          host struct, filled on success
 * Device-side validation failures set MSA_ERR_BAD_Q2K / MSA_ERR_BAD_OFFSETS in
 * the status word (see msa_read_status); forward and backward then do no work.
 */
msa_status msa_build_plan(const int32_t* q2k, const int32_t* doc_offsets, int64_t T,
                          int32_t num_docs, const msa_plan_options* opts, void* workspace,
                          size_t workspace_bytes, msa_stream_t stream, msa_plan* out);

/*
 * msa_build_plan with the plan tables in device memory owned by the library,
 * for callers that cannot allocate device memory where they need a plan (a
 * memory manager that forbids allocation at that point, a hook that is handed
 * only the input buffers).  The pages have no counterpart of this call.
 *   - The tables live in one static 16 MiB device array that every GPU which
 *     loads the library keeps until the process exits.  A problem is
 *     accepted while msa_plan_workspace_bytes(T, num_docs) <= 16 MiB (about
 *     T <= 21400 tokens, a little more or less with the number of
 *     documents); larger ones are rejected with MSA_ERR_WORKSPACE after the
 *     argument checks and before any CUDA call.
 *   - Each call looks the array's device address up on the current device
 *     (cudaGetSymbolAddress); the first call on a device initialises the
 *     library's module there, so make it before any stream capture.
 *   - Every call reuses the same array: the returned plan is valid until the
 *     next msa_build_plan_static call on that device, and calls (or uses of
 *     the plan) that overlap on the GPU race.  Nothing else is allocated.
 * Arguments, validation and errors otherwise as msa_build_plan.
 */
msa_status msa_build_plan_static(const int32_t* q2k, const int32_t* doc_offsets, int64_t T,
                                 int32_t num_docs, const msa_plan_options* opts,
                                 msa_stream_t stream, msa_plan* out);

/* Bytes of forward workspace for a plan (host only).  Dominated by the fp32
 * O pool, T x 64 x 128 x 4 bytes. */
msa_status msa_forward_workspace_bytes(const msa_plan* plan, size_t* bytes);

/*
 * Forward (the pages' flat sparse forward: O [T,64,128] and LSE [T,64]).
 *   q  device bf16 [T,64,128]; k, v device bf16 [T,4,128]
 *   softmax_scale   e.g. 1/sqrt(128)
 *   o   device bf16 [T,64,128] (written)
 *   lse device fp32 [T,64] natural-log LSE (written; -inf for keyless rows)
 *   workspace device, >= msa_forward_workspace_bytes(plan)
 */
msa_status msa_forward(const msa_plan* plan, const void* q, const void* k, const void* v,
                       float softmax_scale, void* o, float* lse, void* workspace,
                       size_t workspace_bytes, msa_stream_t stream);

/* Bytes of backward workspace for a plan (host only). */
msa_status msa_backward_workspace_bytes(const msa_plan* plan, size_t* bytes);

/*
 * Backward (the pages' launch sequence: delta = rowsum(dO * O) -> zero the
 * gradient pools -> main KV-parallel backward -> BF16 finalize), see
 * msa_backward_sm100 run_backward.  O and LSE are the forward's outputs.
 *   dq device bf16 [T,64,128]; dk, dv device bf16 [T,4,128] (written; compact
 *   token order, zero for rows that receive no gradient)
 */
msa_status msa_backward(const msa_plan* plan, const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* dout, float softmax_scale,
                        void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                        msa_stream_t stream);

/* Synchronises the stream and returns the plan's device status (MSA_OK if no
 * device-side error was recorded): the lowest-numbered error, else
 * MSA_ERR_RANGE if the last backward's FP16 dQ pool overflowed.  For tests
 * and diagnostics. */
msa_status msa_read_status(const msa_plan* plan, msa_stream_t stream);

/* Plan counts after synchronising the stream: counts[0] = key blocks NB,
 * [1] = CSR entries, [2] = tasks, [3] = attended (query, head, key) triples,
 * [4] = count entries, [5] = octet-group items, [6] = tasks of the forward's
 * pooled list.  Host array of 7 int64. */
msa_status msa_plan_counts(const msa_plan* plan, msa_stream_t stream, int64_t* counts);

/*
 * Copy the plan tables to host memory after synchronising the stream (for
 * the bit-exact plan tests).  Each destination may be NULL to skip it.
 *   col   int32 [nnz]  query tokens, grouped by task order
 *   tasks int32 [ntasks][4]: {first col index, first key token,
 *         key count | query count << 8 | index head << 12,
 *         index head * nb_cap + global key block}
 * Capacities are element counts; too small -> MSA_ERR_INVALID_ARG.
 */
msa_status msa_plan_export(const msa_plan* plan, msa_stream_t stream, int32_t* col,
                           int64_t col_capacity, int32_t* tasks, int64_t task_capacity);

/*
 * Copy the forward's octet-group tables to host memory after synchronising
 * the stream (for the plan tests).  Each destination may be NULL to skip it.
 *   grouped uint8 [4][T]: 1 where the token's octet is grouped
 *   items   int32 [n_items][36]: first token of octet A, of octet B (-1 if
 *           none), queries of A | of B << 4 | index head << 8 | blocks << 12
 *           | dense << 20, document index, then for a uniform item the
 *           blocks ascending, -1 padded to 32 words, for a dense one (blocks
 *           0 .. b) each token's 64-bit block mask as a low and a high word
 *           (tokens of A, then of B; 32 words); items are ordered by
 *           decreasing work (blocks x octets)
 *   ftasks  int32 [n_ftasks][4]: the task records (as in msa_plan_export) of
 *           the tasks with at least one ungrouped query, in task order
 * Capacities are element counts of the first dimension (T for grouped, which
 * must be >= T); too small -> MSA_ERR_INVALID_ARG.
 */
msa_status msa_plan_export_groups(const msa_plan* plan, msa_stream_t stream, uint8_t* grouped,
                                  int64_t grouped_capacity, int32_t* items,
                                  int64_t item_capacity, int32_t* ftasks,
                                  int64_t ftask_capacity);

/*
 * Compaction of padded packed rows into the compact THD layout, and back
 * (the steps either side of the operation when documents arrive packed into
 * fixed-length rows with trailing padding: NeMo-Automodel PR "feat(minimax-m3):
 * add SM100 MSA sparse attention with custom backward", section "Design" -
 * padding tokens are dropped before the flat attention call and the output is
 * scattered back).  The pages print no interface for them; these are plain
 * row gathers.
 *
 *   x        [B][S][row_bytes] bytes, row b's tokens 0..row_len[b]-1 are real
 *   row_len  int32 [B] device; each value must lie in [0, S] (values outside
 *            are clamped into it)
 *   y        [T][row_bytes] bytes, T = sum of row_len, rows in (b, s) order
 *   row_offsets int32 [B+1] device: exclusive prefix sum of row_len
 *            (written by msa_pack_thd, read by msa_unpack_bshd)
 * row_bytes must be a positive multiple of 16 and all pointers 16-byte
 * aligned; B >= 1, S >= 1, B * S < 2^31.  The caller sizes y for T rows (it
 * knows the lengths; T <= B * S always suffices).  msa_unpack_bshd writes
 * zeros into the padding rows of x.  Both are asynchronous on the stream.
 * Errors: MSA_ERR_INVALID_ARG (null pointer, bad sizes), MSA_ERR_ALIGNMENT,
 * MSA_ERR_CUDA (launch failure).
 */
msa_status msa_pack_thd(const void* x, int32_t B, int32_t S, int32_t row_bytes,
                        const int32_t* row_len, void* y, int32_t* row_offsets,
                        msa_stream_t stream);
msa_status msa_unpack_bshd(const void* y, int32_t B, int32_t S, int32_t row_bytes,
                           const int32_t* row_len, const int32_t* row_offsets, void* x,
                           msa_stream_t stream);

/*
 * Block selection: the index scorer and top-16 choice that produce q2k (the
 * step upstream of the plan: NeMo-Automodel PR "feat(minimax-m3): add SM100
 * MSA sparse attention with custom backward", sections "Summary" and
 * "Design" - an indexer picks, per query and index head, the top-16
 * document-local key blocks).  The pages give no scoring formula; this call
 * implements the plainest reading:
 *   summary(g, d, v) = mean of the index keys ik[j, g, :] of document block v
 *   score(t, g, v)   = dot(iq[t, g, :], summary(g, d, v))  for v = 0 .. b,
 * b = the query's own block.  With b + 1 <= 16 all candidates are selected;
 * otherwise the 16 best by (score descending, block ascending), and with
 * force_local != 0 blocks 0 and b are always kept (plus the 14 best of
 * 1 .. b-1).  Slots hold the blocks in ascending order, then -1.  Scores are
 * fp32: block sums key by key divided by the key count, dot products channel
 * by channel with fused multiply-adds (a fixed order, so the ranking is
 * reproducible).
 *   iq, ik       bf16 [T][4][dim] device, dim in {8, 16, ..., 128}; finite
 *   doc_offsets  int32 [num_docs+1] device, valid as for msa_build_plan
 *   q2k          int32 [4][T][16] device (output)
 *   workspace    msa_select_workspace_bytes(T, num_docs, dim) bytes, 16-byte
 *                aligned (block summaries)
 * Asynchronous on the stream.  Errors: MSA_ERR_INVALID_ARG, MSA_ERR_ALIGNMENT,
 * MSA_ERR_WORKSPACE, MSA_ERR_CUDA.
 */
msa_status msa_select_workspace_bytes(int64_t T, int32_t num_docs, int32_t dim, size_t* bytes);
msa_status msa_select_blocks(const void* iq, const void* ik, int64_t T, int32_t dim,
                             const int32_t* doc_offsets, int32_t num_docs, int32_t force_local,
                             int32_t* q2k, void* workspace, size_t workspace_bytes,
                             msa_stream_t stream);

/*
 * Kernel timing for benchmarks.  While enabled, every kernel the library
 * launches is bracketed by CUDA events on its launch stream.  msa_profile_read
 * synchronises and returns, for the kernel family named (e.g. "fwd_main",
 * "bwd_main"), the launch count and the summed device time since the last
 * reset.  msa_launch_count returns the number of kernels the library has
 * launched since it was loaded.
 */
msa_status msa_profile_enable(int32_t on);
msa_status msa_profile_reset(void);
msa_status msa_profile_read(const char* name, int64_t* launches, double* total_ms);
int64_t msa_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MSA_H_ */
