/*
 * libdspark -- the DSpark per-cycle draft step on one GB300 (sm_103a).
 *
 * Three operations, each a hand-written CUDA kernel:
 *   dspark_markov_draft  the sequential Markov block-draft sampler
 *   dspark_conf_probe    the proposer's Q8_0 confidence probe and its gate
 *   dspark_ws_matvec     the weight-stationary small-M fp16 projection matvec
 *   dspark_ws_matvec_q8  the same matvec over Q8_0 weights (after dspark_q8_0_repack)
 *
 * Conventions shared by every entry point
 *   - Tensor pointers are DEVICE pointers (cudaMalloc / PyTorch allocations), owned
 *     by the caller, row-major and contiguous.  The library never allocates, copies
 *     to the host or synchronizes in these calls: work is enqueued on `stream`
 *     (a cudaStream_t; NULL means the legacy default stream) and the call returns.
 *   - The return value reports argument checking and launch errors only.  Faults
 *     that can only be seen on the device (an out-of-range prev or d2t entry, a
 *     device-side wait that gave up) are recorded in the workspace and reported by
 *     dspark_markov_status() / dspark_ws_matvec_status().
 *   - dspark_last_error() returns a message for the last non-OK status returned on
 *     the calling thread.  No call aborts, exits or traps.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *dspark_stream_t;

typedef enum dspark_status {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID = 1,     /* null pointer, negative or inconsistent size, misalignment */
    DSPARK_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels implement */
    DSPARK_ERR_CUDA = 3,        /* a CUDA runtime call failed (message in dspark_last_error) */
    DSPARK_ERR_TIMEOUT = 4,     /* a device-side wait hit its time limit; outputs undefined */
    DSPARK_ERR_INDEX = 5        /* a prev or d2t entry was out of range; those ids are -1 */
} dspark_status;

/* Message for the last non-OK status on this thread ("" if none).  Thread-local storage
 * owned by the library; valid until the next call on the same thread. */
const char *dspark_last_error(void);

/* Library version string, e.g. "libdspark 0.1 sm_103a". */
const char *dspark_version(void);

/* =====================================================================================
 * Markov block draft
 *
 * Source: vllm.cpp issue #436 "SPEC-DSPARK W7: the sequential Markov sample loop is
 * HOST-side", section "The fix" (per-step chain, lowest-index tie-break, identity d2t,
 * prev kept on the device, only the final ids read back) and "W7 LANDED"
 * (markov_w2 is [draft_vocab, markov_rank] bf16 and is re-read whole every step).
 *
 * For every request r and draft position i = 0 .. k-1, with p = prev[r] at i = 0:
 *   h        = markov_w1[p, :]                                  (gather)
 *   bias[v]  = sum_j markov_w2[v, j] * h[j]                     (bias GEMV, fp32 accumulate)
 *   logit[v] = base_logits[r, i, v] + bias[v]                   (fp32)
 *   id       = smallest v attaining max_v logit[v]               (greedy argmax)
 *   out_ids[r, i] = d2t ? d2t[id] : id                          (target-space id)
 *   p        = id                                               (draft-space id)
 *
 * Arguments
 *   base_logits  float  [num_reqs, k, vocab]
 *   markov_w1    bf16   [vocab, rank] (raw 16-bit patterns)
 *   markov_w2    bf16   [vocab, rank]; 16-byte aligned
 *   d2t          int32  [vocab] draft->target map, or NULL for the identity
 *   prev         int64  [num_reqs]; in: previous draft id per request,
 *                out: the last draft-space id of each request (written at the end)
 *   out_ids      int64  [num_reqs, k] target-space draft ids
 *   dbg_logits   float  [num_reqs, k, vocab] or NULL: every logit (tests only; costs
 *                bandwidth)
 *   dbg_bias     float  [num_reqs, k, vocab] or NULL: every bias value (tests only)
 *   workspace    device scratch of at least dspark_markov_workspace_bytes() bytes,
 *                256-byte aligned; it also holds the device status word.  Calls that
 *                share one workspace must not overlap on the device.
 * Supported: rank in {64, 128, 256}; 1 <= num_reqs <= 8; vocab >= 1;
 *   k >= 0 (k == 0 or num_reqs == 0 enqueues nothing).
 * Device-side errors: a prev entry outside [0, vocab) or a negative d2t entry makes
 *   the affected ids -1 and sets DSPARK_ERR_INDEX in the status word.
 * Two kernels compute this, with the same tensor-core instructions for every bias value,
 *   so they give bit-identical logits and ids; the call picks one from the sizes:
 *   - single-cluster: for num_reqs <= 2 when markov_w1 and markov_w2 (and the exchange
 *     buffers) fit in the shared memory of one thread-block cluster of up to 16 CTAs (about
 *     vocab <= 12 K at rank 64, <= 6 K at rank 128, <= 2 K at rank 256), vocab is a multiple
 *     of 4 and base_logits is 16-byte aligned: one cluster launch that keeps both matrices on
 *     chip and passes each position's argmax and the winner's markov_w1 row through
 *     distributed shared memory.  The kernel resets the status word itself.
 *   - grid: otherwise, one cooperative kernel launch (at most one CTA per SM) preceded by
 *     a memset of the workspace header.
 *   Either can be captured in a CUDA graph.
 * ===================================================================================== */
size_t dspark_markov_workspace_bytes(int num_reqs, int k, int vocab, int rank);

dspark_status dspark_markov_draft(const float *base_logits, const uint16_t *markov_w1,
                                  const uint16_t *markov_w2, const int32_t *d2t, int64_t *prev,
                                  int num_reqs, int k, int vocab, int rank, int64_t *out_ids,
                                  float *dbg_logits, float *dbg_bias, void *workspace,
                                  size_t workspace_bytes, dspark_stream_t stream);

/* The same draft with the kernel named explicitly: DSPARK_MARKOV_KERNEL_AUTO (what
 * dspark_markov_draft does), DSPARK_MARKOV_KERNEL_GRID or DSPARK_MARKOV_KERNEL_CLUSTER (any
 * num_reqs, where its shared memory fits).  Asking for the single-cluster kernel where it
 * does not fit returns DSPARK_ERR_UNSUPPORTED and enqueues nothing; any other value is
 * DSPARK_ERR_INVALID. */
#define DSPARK_MARKOV_KERNEL_AUTO 0
#define DSPARK_MARKOV_KERNEL_GRID 1
#define DSPARK_MARKOV_KERNEL_CLUSTER 2
dspark_status dspark_markov_draft_kernel(const float *base_logits, const uint16_t *markov_w1,
                                         const uint16_t *markov_w2, const int32_t *d2t,
                                         int64_t *prev, int num_reqs, int k, int vocab, int rank,
                                         int64_t *out_ids, float *dbg_logits, float *dbg_bias,
                                         void *workspace, size_t workspace_bytes, int kernel,
                                         dspark_stream_t stream);

/* The kernel dspark_markov_draft uses on the current device for these sizes and a 16-byte
 * aligned base_logits: DSPARK_MARKOV_KERNEL_GRID or DSPARK_MARKOV_KERNEL_CLUSTER.  Host
 * only; may query the device's cluster occupancy once. */
int dspark_markov_kernel_for(int num_reqs, int k, int vocab, int rank);

/* Synchronizes `stream`, then reads the status word that the last dspark_markov_draft
 * on `workspace` left: DSPARK_OK, DSPARK_ERR_INDEX or DSPARK_ERR_TIMEOUT. */
dspark_status dspark_markov_status(const void *workspace, dspark_stream_t stream);

/* Fault-injection hook for testing the device-side wait limit: the same launch as
 * dspark_markov_draft with the grid kernel (whatever the sizes), except that its grid-wide
 * step barrier expects `missing_arrivals` more arrivals than there are CTAs (so with
 * missing_arrivals > 0
 * it can never complete) and every device-side wait gives up after `timeout_us`
 * microseconds.  The kernel then records DSPARK_ERR_TIMEOUT, drains its in-flight
 * copies and returns; nothing hangs.  Not for production use. */
dspark_status dspark_markov_draft_debug(const float *base_logits, const uint16_t *markov_w1,
                                        const uint16_t *markov_w2, const int32_t *d2t,
                                        int64_t *prev, int num_reqs, int k, int vocab, int rank,
                                        int64_t *out_ids, void *workspace,
                                        size_t workspace_bytes, unsigned missing_arrivals,
                                        unsigned timeout_us, dspark_stream_t stream);

/* Plan form: records one dspark_markov_draft call (fixed pointers and sizes) into an
 * instantiated CUDA graph, so that each draft is a single graph launch.  Creation
 * captures on a private stream and may allocate host/driver objects; launching
 * allocates nothing.  The tensors must stay alive while the plan is used. */
typedef struct dspark_markov_plan dspark_markov_plan;

dspark_status dspark_markov_plan_create(const float *base_logits, const uint16_t *markov_w1,
                                        const uint16_t *markov_w2, const int32_t *d2t,
                                        int64_t *prev, int num_reqs, int k, int vocab,
                                        int rank, int64_t *out_ids, void *workspace,
                                        size_t workspace_bytes, dspark_markov_plan **plan_out);
dspark_status dspark_markov_plan_launch(dspark_markov_plan *plan, dspark_stream_t stream);
void dspark_markov_plan_destroy(dspark_markov_plan *plan);

/* Allocation-free Markov draft.  The paper has no counterpart: this entry point exists
 * for callers that cannot call cudaMalloc or hand over device scratch -- for example a
 * plugin inside a host engine whose device memory is owned by the engine's allocator, or
 * a latency-critical loop where cudaMalloc's implicit device synchronization is not
 * acceptable.  It computes exactly what dspark_markov_draft computes (same kernel, same
 * arguments except the workspace and the debug outputs) and calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *   Scratch: a 4352-byte array in the library's static device memory (enough for
 *   k <= 64 positions; larger k is rejected with DSPARK_ERR_UNSUPPORTED).  Every GPU that
 *   loads the library holds its own copy until the process exits.  Each call clears it
 *   (a memset on `stream`) before the kernel.  All calls on one device share that copy:
 *   calls that overlap on the GPU (for example on two streams with no ordering between
 *   them) race and give undefined results, so serialize them.
 *   Errors seen only on the device: the status word lives in the same array and cannot be
 *   read by the caller.  Instead, out_ids is set to -1 (a memset on `stream`) before the
 *   kernel, so a position the kernel did not finish -- a device-side wait that gave up, or
 *   an out-of-range prev / d2t entry -- reads -1; prev is only written when every position
 *   finished.  Treat a draft with any -1 id as failed.
 *   Set-up: the array's device address is looked up with cudaGetSymbolAddress the first
 *   time a CUDA context (normally: once per device, with that device current) uses this
 *   entry point, and cached with that context's id; a later context on the same device
 *   (one the caller created, or the primary context after cudaDeviceReset) gets its own
 *   lookup.  The first lookup may load the library's device code: make the first call in
 *   each context before any stream capture. */
dspark_status dspark_markov_draft_noalloc(const float *base_logits, const uint16_t *markov_w1,
                                          const uint16_t *markov_w2, const int32_t *d2t,
                                          int64_t *prev, int num_reqs, int k, int vocab, int rank,
                                          int64_t *out_ids, dspark_stream_t stream);

/* =====================================================================================
 * Confidence probe
 *
 * Source: ds4 PR #772 "dspark: cut per-cycle CUDA overheads (single-draft decode, GPU
 * confidence probe)", sections "Summary" and "Root cause": a 7424-wide matvec of the
 * hidden state against Q8_0 weights, evaluated on the GPU with a 4-byte readback; the
 * result only gates the proposal length.
 *
 * For each probe p:
 *   z[p]    = bias + sum_b d_b * sum_{j<32} q_{b,j} * hidden[p, 32b + j]
 *   gate[p] = (sigmoid(z[p]) >= threshold), computed as z[p] >= log(t / (1 - t))
 *
 * Arguments
 *   w_q8_0     K/32 Q8_0 blocks of 34 bytes each: fp16 scale d (little endian) followed
 *              by 32 int8 values q; any byte alignment
 *   hidden     float [n_probes, K]; 16-byte aligned
 *   bias       scalar added to every probe's dot product
 *   threshold  in (0, 1)
 *   K          > 0, multiple of 32
 *   n_probes   >= 0 (0 enqueues nothing); probes are independent.  Small batches run one
 *              CTA per probe; batches larger than 8 x the SM count run on persistent CTAs
 *              that stream the hidden rows through a ring of bulk copies.  Every probe gives
 *              the same bits either way.
 *   logit_out  float [n_probes] or NULL
 *   gate_out   int32 [n_probes]: 1 = keep drafting, 0 = stop; -1 (with a NaN logit) only if
 *              a device-side wait of the large-batch form gave up, which does not happen in
 *              normal operation.  May be device memory or mapped pinned host memory (then
 *              the 4-byte readback is the kernel's own store).  Must not be NULL.
 * ===================================================================================== */
dspark_status dspark_conf_probe(const void *w_q8_0, const float *hidden, float bias,
                                float threshold, int K, int n_probes, float *logit_out,
                                int32_t *gate_out, dspark_stream_t stream);

/* The same probe over an input that arrives in two pieces, e.g. the hidden state and the
 * Markov state kept in separate buffers (ds4 PR #772, "Summary": the probe reads the hidden
 * copy and the markov_state).  Probe p's input vector is
 *   [hidden[p * ld_hidden + 0 .. K_hidden); state[p * ld_state + 0 .. K_state)]
 * and the Q8_0 row covers K_hidden + K_state elements.  K_hidden > 0 and K_state >= 0 are
 * multiples of 4 with a sum that is a multiple of 32; hidden and state are 16-byte aligned,
 * ld_* are multiples of 4 and at least the widths.  The result is bit-identical to
 * dspark_conf_probe on the concatenated vector. */
dspark_status dspark_conf_probe_split(const void *w_q8_0, const float *hidden, int K_hidden,
                                      long long ld_hidden, const float *state, int K_state,
                                      long long ld_state, float bias, float threshold, int n_probes,
                                      float *logit_out, int32_t *gate_out, dspark_stream_t stream);

/* =====================================================================================
 * Weight-stationary small-M matvec
 *
 * Source: SharpInference issue #441 "DSpark GPU draft round runs ~3x the bandwidth
 * floor -- small-M (B=7) projection GEMMs -> weight-stationary matvec", sections
 * "Observation", "Hypothesis" and "Proposed work": fp16 projections with M = B = 7
 * rows where each weight element should be read from HBM once for all rows.
 *
 *   Y[m, n] = sum_k X[m, k] * W[n, k]      (fp16 inputs, fp32 accumulation)
 *
 * Runs on the tcgen05 tensor cores (128 weight rows x 16 padded activation rows per MMA).
 * K may be split over S = 2, 4 or 8 CTAs per 128-row block (chosen from N, K and the SM
 * count); they form a thread-block cluster and their fp32 partial sums are added in
 * distributed shared memory in a fixed order, 0 + p_0 + ... + p_{S-1}.
 *
 * Arguments
 *   W          fp16 [N, K] (out x in), 16-byte aligned
 *   X          fp16 [M, K], 16-byte aligned
 *   Y          [M, N]: fp32 if y_is_fp32, else fp16 rounded to nearest even
 *   workspace  device scratch of at least dspark_ws_matvec_workspace_bytes(M, N, K)
 *              bytes (256), 256-byte aligned, ZERO-FILLED before its first use: it holds
 *              the device status word (see dspark_ws_matvec_status).  Calls sharing a
 *              workspace must not overlap on the device.
 *   Supported: 1 <= M <= 16, N >= 1, K >= 8 with K % 8 == 0 (M == 0 or N == 0
 *   enqueues nothing).  The result of row m does not depend on M: every output is
 *   summed in one fixed order.
 * ===================================================================================== */
size_t dspark_ws_matvec_workspace_bytes(int M, int N, int K);

dspark_status dspark_ws_matvec(const uint16_t *W, const uint16_t *X, void *Y, int y_is_fp32,
                               int M, int N, int K, void *workspace, size_t workspace_bytes,
                               dspark_stream_t stream);

/* Grouped form: up to 8 independent problems (e.g. the q, k and v projections of a layer,
 * or gate and up) in one launch, so their fixed launch and pipeline costs are paid once and
 * the SMs left idle by one problem's tail take the next one's units.  Each problem has the
 * arguments and limits of dspark_ws_matvec; its results are bit-identical to a separate
 * dspark_ws_matvec call.  Problems with M == 0 or N == 0 are skipped.  The workspace
 * (dspark_ws_matvec_grouped_workspace_bytes(problems, n), zero-filled before first use) holds
 * the status word, as for dspark_ws_matvec.  More than 8 problems: DSPARK_ERR_UNSUPPORTED. */
typedef struct dspark_ws_problem {
    const uint16_t *W;  /* fp16 [N, K] */
    const uint16_t *X;  /* fp16 [M, K] */
    void *Y;            /* [M, N], fp32 if y_is_fp32 else fp16 */
    int y_is_fp32;
    int M, N, K;
} dspark_ws_problem;

size_t dspark_ws_matvec_grouped_workspace_bytes(const dspark_ws_problem *problems, int n_problems);
dspark_status dspark_ws_matvec_grouped(const dspark_ws_problem *problems, int n_problems,
                                       void *workspace, size_t workspace_bytes,
                                       dspark_stream_t stream);

/* Synchronizes `stream`, then reads the status word of a dspark_ws_matvec or
 * dspark_ws_matvec_q8 workspace (its first 4 bytes): DSPARK_OK, or DSPARK_ERR_TIMEOUT if a
 * device-side wait of a call on it gave up since the last check (the kernel then skipped
 * the affected outputs and returned).  A reported timeout is cleared, leaving the status
 * word zero again. */
dspark_status dspark_ws_matvec_status(void *workspace, dspark_stream_t stream);

/* Fault-injection hook for testing the device-side wait limit: the same launch as
 * dspark_ws_matvec, except that the epilogue first waits `stall_us` microseconds on a
 * barrier that nothing signals; the wait gives up, the kernel records DSPARK_ERR_TIMEOUT in
 * the workspace status word and finishes normally.  Not for production use. */
dspark_status dspark_ws_matvec_debug(const uint16_t *W, const uint16_t *X, void *Y, int y_is_fp32,
                                     int M, int N, int K, void *workspace, size_t workspace_bytes,
                                     unsigned stall_us, dspark_stream_t stream);

/* =====================================================================================
 * Weight-stationary small-M matvec with Q8_0 weights
 *
 * Source: SharpInference issue #441, "Proposed work": the weight-stationary kernels it
 * reuses read quantized weights, and a structure-of-arrays repack of the quantized blocks
 * may be needed.  Q8_0 (ggml): per 32 consecutive weights of a row, one fp16 scale d and 32
 * int8 values q; the weight is d * q.
 *
 *   Y[m, n] = sum_b d[n, b] * sum_{j<32} q[n, 32b + j] * X[m, 32b + j]   (fp32 accumulation)
 *
 * dspark_q8_0_repack turns the ggml array of 34-byte blocks (row-major by weight row: the
 * K/32 blocks of row 0, then row 1, ...) into the two arrays dspark_ws_matvec_q8 reads:
 *   q  int8 [N, K]      the quantized values, 16-byte aligned
 *   d  fp16 [N, K/32]   the block scales (bit patterns), 16-byte aligned for the matvec
 * Supported: K % 32 == 0 (N == 0 enqueues nothing).
 *
 * dspark_ws_matvec_q8 runs on the tcgen05 tensor cores: q (exact in fp16) times X gives, per
 * Q8_0 block, an fp32 partial sum that the kernel then scales by d in fp32, so the dequantized
 * weight d * q is never rounded to a 16-bit type.
 *   X          fp16 [M, K], 16-byte aligned
 *   Y          [M, N]: fp32 if y_is_fp32, else fp16 rounded to nearest even
 *   workspace  device scratch of at least dspark_ws_matvec_q8_workspace_bytes(M, N, K) bytes
 *              (256), 256-byte aligned and ZERO-FILLED before its first use: it holds the
 *              device status word.  Calls sharing a workspace must not overlap on the device.
 *   K is split over S <= 8 CTAs per 128-row block when there are at most as many row blocks
 *   as SMs; the S CTAs form a thread-block cluster and add their partial sums in distributed
 *   shared memory in a fixed order.
 *   Supported: 1 <= M <= 16, N >= 1, K a positive multiple of 256 (M == 0 or N == 0 enqueues
 *   nothing).  Every output is summed in one fixed order, so row m's result does not depend
 *   on M.
 * ===================================================================================== */
dspark_status dspark_q8_0_repack(const void *w_q8_0, int8_t *q, uint16_t *d, int N, int K,
                                 dspark_stream_t stream);

size_t dspark_ws_matvec_q8_workspace_bytes(int M, int N, int K);

dspark_status dspark_ws_matvec_q8(const int8_t *Wq, const uint16_t *Wd, const uint16_t *X, void *Y,
                                  int y_is_fp32, int M, int N, int K, void *workspace,
                                  size_t workspace_bytes, dspark_stream_t stream);

/* Grouped form: up to 8 independent Q8_0 problems in one launch (e.g. the four projections
 * of a layer), so the fixed launch and pipeline costs are paid once and no SM idles while
 * another finishes a long row block.  Each problem has the arguments and limits of
 * dspark_ws_matvec_q8.  The 128-row blocks of all problems, each over all of K, form one
 * sequence of 256-k superblocks that min(SMs, superblocks) co-resident CTAs (a cooperative
 * launch) take in equal contiguous ranges (stream-K); a row block cut by a range boundary is
 * finished by the CTA holding its first superblocks, which adds the partial sums of the CTAs
 * after it in CTA order.  Every output is summed in one fixed order, so results are
 * deterministic; they can differ in the last bits from a separate dspark_ws_matvec_q8 call,
 * which splits K differently.  Problems with M == 0 or N == 0 are skipped; with only one
 * problem left the call is a dspark_ws_matvec_q8 call.  The workspace
 * (dspark_ws_matvec_q8_grouped_workspace_bytes on the device that runs the call: a status
 * word, one flag and 8 KB of partial sums per SM) must be zero-filled before its first use;
 * the kernel leaves the flags zero again, except after a wait that gave up
 * (DSPARK_ERR_TIMEOUT), after which the workspace must be zero-filled again.  More than 8
 * problems: DSPARK_ERR_UNSUPPORTED. */
typedef struct dspark_ws_q8_problem {
    const int8_t *Wq;    /* int8 [N, K] (dspark_q8_0_repack), 16-byte aligned */
    const uint16_t *Wd;  /* fp16 [N, K/32] scales, 16-byte aligned */
    const uint16_t *X;   /* fp16 [M, K], 16-byte aligned */
    void *Y;             /* [M, N], fp32 if y_is_fp32 else fp16 */
    int y_is_fp32;
    int M, N, K;
} dspark_ws_q8_problem;

size_t dspark_ws_matvec_q8_grouped_workspace_bytes(const dspark_ws_q8_problem *problems,
                                                   int n_problems);
dspark_status dspark_ws_matvec_q8_grouped(const dspark_ws_q8_problem *problems, int n_problems,
                                          void *workspace, size_t workspace_bytes,
                                          dspark_stream_t stream);

/* Fault-injection hook for testing the grouped launch's wait on another CTA: the same launch
 * as dspark_ws_matvec_q8_grouped (at least two non-empty problems, else DSPARK_ERR_INVALID),
 * except that every wait of the kernel gives up after `timeout_us` microseconds instead of
 * 2 s, and CTA `withheld_cta` writes its partial sums but never sets its flag.  If that
 * CTA's range starts inside a row block, the CTA finishing the row block waits for the flag,
 * gives up, skips that row block's outputs and records DSPARK_ERR_TIMEOUT in the workspace
 * status word (dspark_ws_matvec_status); the workspace must then be zero-filled again.  Any
 * other CTA number gives the ordinary result.  Not for production use. */
dspark_status dspark_ws_matvec_q8_grouped_debug(const dspark_ws_q8_problem *problems, int n_problems,
                                                void *workspace, size_t workspace_bytes,
                                                int withheld_cta, unsigned timeout_us,
                                                dspark_stream_t stream);

/* As dspark_ws_matvec_debug, for the Q8_0 matvec (status read by dspark_ws_matvec_status). */
dspark_status dspark_ws_matvec_q8_debug(const int8_t *Wq, const uint16_t *Wd, const uint16_t *X,
                                        void *Y, int y_is_fp32, int M, int N, int K,
                                        void *workspace, size_t workspace_bytes, unsigned stall_us,
                                        dspark_stream_t stream);

/* =====================================================================================
 * Host-buffer forms
 *
 * The three operations above with their per-call inputs read from host memory and their
 * outputs written to host memory: the host-to-device copies, the same kernel, and the
 * device-to-host copies are enqueued in that order on `stream` (cudaMemcpyAsync), so a cycle
 * that starts from host data is one call per operation and one stream synchronization.
 * Resident tensors (markov_w1/w2, d2t, the Q8_0 probe row, projection weights) stay device
 * pointers.  Host buffers should be page-locked for the copies to be asynchronous.  Results
 * are bit-identical to the device-pointer forms.
 *
 * device_scratch: caller-owned device memory of at least the matching *_scratch_bytes(),
 * 256-byte aligned; it holds the device copies of the inputs and outputs and the operation's
 * workspace.  For dspark_ws_matvec_host the scratch must be ZERO-FILLED before first use
 * (its first part is the matvec workspace with its status word).  Calls
 * sharing a scratch must not overlap on the device.
 *
 *   dspark_markov_draft_host: base_host float [num_reqs, k, vocab]; prev_host int64
 *     [num_reqs] in/out (read before the draft, overwritten with each request's last draft
 *     id); out_ids_host int64 [num_reqs, k].
 *   dspark_conf_probe_host: hidden_host float [n_probes, K]; gate_host int32 [n_probes];
 *     logit_host float [n_probes] or NULL.
 *   dspark_ws_matvec_host: X_host fp16 [M, K]; Y_host [M, N] fp32 if y_is_fp32 else fp16.
 * inputs_copied: optional cudaEvent_t (NULL for none) recorded on `stream` right after the
 *   host-to-device copies.  Pinned copies queued on several streams are served in the order
 *   they become ready, not interleaved; a caller overlapping two operations can make the
 *   second one's stream wait on the first one's event so a small input is not queued behind
 *   a large one.
 * Argument errors are reported before anything is enqueued; a *_scratch_bytes() of 0 means
 * the sizes are invalid (or, for the matvec, that no CUDA device could be queried).
 * ===================================================================================== */
size_t dspark_markov_draft_host_scratch_bytes(int num_reqs, int k, int vocab, int rank);
dspark_status dspark_markov_draft_host(const float *base_host, const uint16_t *markov_w1,
                                       const uint16_t *markov_w2, const int32_t *d2t,
                                       int64_t *prev_host, int num_reqs, int k, int vocab, int rank,
                                       int64_t *out_ids_host, void *device_scratch,
                                       size_t scratch_bytes, void *inputs_copied,
                                       dspark_stream_t stream);

size_t dspark_conf_probe_host_scratch_bytes(int K, int n_probes);
dspark_status dspark_conf_probe_host(const void *w_q8_0, const float *hidden_host, float bias,
                                     float threshold, int K, int n_probes, float *logit_host,
                                     int32_t *gate_host, void *device_scratch, size_t scratch_bytes,
                                     void *inputs_copied, dspark_stream_t stream);

size_t dspark_ws_matvec_host_scratch_bytes(int M, int N, int K);
dspark_status dspark_ws_matvec_host(const uint16_t *W, const uint16_t *X_host, void *Y_host,
                                    int y_is_fp32, int M, int N, int K, void *device_scratch,
                                    size_t scratch_bytes, void *inputs_copied,
                                    dspark_stream_t stream);

/* Grouped host-buffer form of dspark_ws_matvec_grouped: in `problems`, W is a device pointer
 * and X / Y are HOST pointers.  All X copies are enqueued first (then inputs_copied is
 * recorded), then the one grouped launch, then the Y copies.  Scratch: at least
 * dspark_ws_matvec_grouped_host_scratch_bytes(problems, n), 256-byte aligned, zero-filled
 * before first use (its first part is the grouped workspace). */
size_t dspark_ws_matvec_grouped_host_scratch_bytes(const dspark_ws_problem *problems,
                                                   int n_problems);
dspark_status dspark_ws_matvec_grouped_host(const dspark_ws_problem *problems, int n_problems,
                                            void *device_scratch, size_t scratch_bytes,
                                            void *inputs_copied, dspark_stream_t stream);

/* =====================================================================================
 * Draft step with device-side base logits
 *
 * Source: vllm.cpp issue #436, "W7 LANDED": the half W7 deferred is a block-forward
 * variant that returns the base logits on the device instead of downloading
 * [num_reqs, k, draft_vocab] floats.  Here the draft head's lm_head projection runs as a
 * weight-stationary matvec (SharpInference issue #441) that writes the fp32 base logits into
 * device memory, followed by the Markov draft; both are recorded into one CUDA graph.
 *
 *   base[r, i, v] = sum_h hidden_states[r * k + i, h] * lm_head[v, h]   (fp32)
 *   then dspark_markov_draft(base, ...)
 *
 * Arguments
 *   lm_head        fp16 [vocab, hidden_dim], 16-byte aligned
 *   hidden_states  fp16 [num_reqs * k, hidden_dim], 16-byte aligned
 *   base_logits    float [num_reqs, k, vocab] device buffer the plan writes and reads
 *   markov_workspace  >= dspark_markov_workspace_bytes(num_reqs, k, vocab, rank)
 *   ws_workspace   >= dspark_ws_matvec_workspace_bytes(num_reqs * k, vocab, hidden_dim),
 *                  zero-filled before first use (see dspark_ws_matvec)
 *   other arguments as for dspark_markov_draft.
 * Supported: num_reqs * k <= 16 (the matvec's row limit), plus the limits of the two calls.
 * ===================================================================================== */
typedef struct dspark_draft_plan dspark_draft_plan;

dspark_status dspark_draft_plan_create(const uint16_t *lm_head, const uint16_t *hidden_states,
                                       int hidden_dim, const uint16_t *markov_w1,
                                       const uint16_t *markov_w2, const int32_t *d2t, int64_t *prev,
                                       int num_reqs, int k, int vocab, int rank, float *base_logits,
                                       int64_t *out_ids, void *markov_workspace,
                                       size_t markov_workspace_bytes, void *ws_workspace,
                                       size_t ws_workspace_bytes, dspark_draft_plan **plan_out);
dspark_status dspark_draft_plan_launch(dspark_draft_plan *plan, dspark_stream_t stream);
void dspark_draft_plan_destroy(dspark_draft_plan *plan);

/* =====================================================================================
 * Confidence-gated draft (decision stays on the device)
 *
 * Source: ds4 PR #772, "Summary" and "Root cause": the confidence probe gates whether the
 * proposer keeps drafting; the PR evaluates it on the GPU but reads the 4-byte decision back.
 * Here one CUDA graph holds the probe (one probe over probe_input[0 .. K)) and a conditional
 * IF node whose body is the Markov draft: the probe kernel sets the condition, so the draft
 * runs only if sigmoid(z) >= threshold, with no host round trip.  gate_out[0] / logit_out[0]
 * still receive the decision and the logit.  When the gate is 0 the draft's outputs (out_ids,
 * prev, the workspace status word) are left untouched.
 * Arguments: the probe's (see dspark_conf_probe, n_probes = 1) followed by the Markov
 * draft's (see dspark_markov_draft, no debug outputs).
 * ===================================================================================== */
typedef struct dspark_gated_plan dspark_gated_plan;

dspark_status dspark_gated_draft_plan_create(const void *w_q8_0, const float *probe_input, int K,
                                             float bias, float threshold, float *logit_out,
                                             int32_t *gate_out, const float *base_logits,
                                             const uint16_t *markov_w1, const uint16_t *markov_w2,
                                             const int32_t *d2t, int64_t *prev, int num_reqs, int k,
                                             int vocab, int rank, int64_t *out_ids, void *workspace,
                                             size_t workspace_bytes, dspark_gated_plan **plan_out);
dspark_status dspark_gated_draft_plan_launch(dspark_gated_plan *plan, dspark_stream_t stream);
void dspark_gated_draft_plan_destroy(dspark_gated_plan *plan);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
