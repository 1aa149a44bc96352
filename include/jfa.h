/*
 * jfa.h -- C ABI of libjfa: Jagged Flash Attention on GB300 (sm_103a).
 *
 * Exact attention O = softmax(scale * Q K^T) V, forward and backward, computed
 * directly on packed variable-length sequences.  Sources (four web pages on the
 * subject):
 *   [C]  "Optimizing Jagged Flash Attention with TLX" (commentary page):
 *        sections "why unequal lengths change the problem", "architecture",
 *        "load balancing", "performance and feature scope".
 *   [N]  n1n.ai page on JFA with TLX: the padded-tensor cost and the jagged
 *        layout example (offsets [0, 128, 4224, 4736, 6784]).
 *   [B]  "TLX Block Attention" (translation of the PyTorch blog): sections 2.1
 *        (the fixed-block simplifications), 3 (warp-specialised pipeline),
 *        4 (backward without a log-sum-exp tensor), 5 (variable-length scheduling).
 *   [R]  aixai.ru summary of the JFA-TLX work: "What is JFA", "Framework",
 *        "Tile balancing and Cluster Launch Control", "dQ epilogue",
 *        "Loop peeling", "Paired CTAs".
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Packed ("jagged") layout [C, N]: the tokens of all sequences are stored
 *    back to back; offsets[b] .. offsets[b+1]-1 are the rows of sequence b,
 *    offsets[0] = 0, offsets has batch+1 int32 entries.
 *  - Tensors are contiguous row-major [rows, heads, head_dim] bf16: element
 *    (t, h, d) is at t*heads*head_dim + h*head_dim + d.  K and V (and dK, dV)
 *    have num_kv_heads heads; query head h reads key/value head
 *    h / (num_heads / num_kv_heads).
 *  - Self-attention (broadcast_q == 0): q, o, dO, dq have offsets[batch] rows.
 *  - Broadcast-Q (broadcast_q != 0) [C "unequal lengths"; R "What is JFA"]:
 *    q and dq have nq_broadcast rows shared by every sequence; o and dO have
 *    batch * nq_broadcast rows (sequence-major: rows b*nq .. b*nq+nq-1 belong to
 *    sequence b); dq is the sum over all sequences.
 *  - lse is fp32 [num_heads, rows of o]: the natural-log log-sum-exp of each
 *    score row, L = m + log(l) [B 2.1, Listing 1].  An empty sequence in
 *    broadcast mode yields o rows of 0 and lse = -inf.
 *  - Causal masking (key j visible to query i iff j <= i inside a sequence) is
 *    supported for self-attention only.
 *  - head_dim must be 64 or 128 (the pages allow up to 128 [C "feature scope"];
 *    this library builds those two).  Grouped-query attention (GQA) is
 *    supported forward and backward.  The pages' own implementation limits
 *    the backward to one group [C "feature scope"]; here dk and dv of key/value
 *    head g sum the gradients of all its query heads.
 *  - offsets_dev is the device copy of the offsets; offsets_host the host copy,
 *    from which all scheduling is planned on the CPU with no device sync
 *    [B 5].  Both must hold the same values; only offsets_host is validated.
 *  - Ownership: the caller owns every buffer, including `workspace` (device
 *    memory of at least jfa_workspace_size() bytes, any contents).  The library
 *    allocates no device memory and keeps no state across calls except cached
 *    device properties and kernel attributes.
 *  - Streams: all device work is enqueued on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  Calls return once the work is enqueued.
 *    The host-side offsets are read before the call returns.
 *  - Not for stream capture: each call plans on the host and copies its plan to
 *    the device from a small ring of host buffers that later calls reuse, so a
 *    captured graph would replay with whatever a buffer then holds.  Do not
 *    call these entry points while `stream` is being captured into a CUDA
 *    graph.
 *  - Errors: every call returns a jfa_status; nothing is thrown across the ABI.
 *    Argument errors are detected before any work is enqueued.  A kernel whose
 *    internal wait times out records JFA_ERR_DEVICE_TIMEOUT in the workspace,
 *    which jfa_device_status() reports.
 */
#ifndef JFA_H_
#define JFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  JFA_OK = 0,
  JFA_ERR_INVALID_ARG = 1,          /* null pointer, negative size, misaligned pointer */
  JFA_ERR_UNSUPPORTED = 2,          /* head_dim not 64/128, causal+broadcast,
                                       num_heads % num_kv_heads != 0, more than
                                       2^31 - 1 broadcast output rows */
  JFA_ERR_BAD_OFFSETS = 3,          /* offsets[0] != 0, decreasing, or a length > max_len */
  JFA_ERR_WORKSPACE_TOO_SMALL = 4,
  JFA_ERR_ARCH = 5,                 /* current device is not compute capability 10.x */
  JFA_ERR_CUDA = 6,                 /* a CUDA runtime call or launch failed */
  JFA_ERR_DEVICE_TIMEOUT = 7,       /* a kernel wait ran out (see jfa_device_status) */
  JFA_ERR_TOO_LARGE = 8             /* jfa_fwd_noalloc: the plan exceeds its static scratch */
} jfa_status;

typedef enum {
  JFA_OP_FWD = 0,
  JFA_OP_BWD = 1,
  JFA_OP_BLOCK_FWD = 2,
  JFA_OP_BLOCK_BWD = 3,
  JFA_OP_TOPK_SELECT = 4,  /* jfa_topk_select (an upper bound with grouped K/V heads) */
  JFA_OP_FWD_TOPK = 5,     /* jfa_fwd_topk */
  JFA_OP_BLOCK_FWD_ROPE = 6, /* block_attn_fwd_rope: + the packed rotary table */
  JFA_OP_BLOCK_BWD_ROPE = 7  /* block_attn_bwd_rope: the same */
} jfa_op;

/*
 * jfa_fwd -- jagged flash-attention forward [C "architecture"; R "Framework";
 * B 2.1 Listing 1 for the online-softmax recurrence; N for the layout].
 *   o   = softmax(scale * q k^T) v per sequence and head (bf16 out),
 *   lse = log-sum-exp per row (fp32, may be NULL to skip writing it).
 * Work is planned on the host: 256-row query units sorted by K/V length,
 * taken in that order under Cluster Launch Control (the default) or dealt to
 * one persistent CTA per SM in snake (zigzag) order under the static schedule
 * [R "Tile balancing and Cluster Launch Control"; jfa_set_schedule].
 */
int jfa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* offsets_dev,
            const int32_t* offsets_host, int batch, int max_len, int nq_broadcast, int num_heads,
            int num_kv_heads, int head_dim, float scale, int causal, int broadcast_q, void* workspace,
            size_t workspace_bytes, void* stream);

/*
 * jfa_bwd -- jagged flash-attention backward [B 4 for the gradient algebra;
 * R "Paired CTAs" (five GEMMs per K/V block), "dQ epilogue"; C "load balancing"].
 * Inputs are the forward's q, k, v, o, lse and the output gradient dO; outputs
 * dq (bf16, like q), dk and dv (bf16, like k):
 *   P = exp(scale q k^T - lse), dV = P^T dO, dP = dO V^T, Di = rowsum(dO o O),
 *   dS = P o (dP - Di), dQ = scale dS K, dK = scale dS^T Q.
 * With GQA, dk and dv of key/value head g are the sums over query heads
 * g*G .. g*G+G-1 (G = num_heads / num_kv_heads), formed in one CTA without
 * atomics.  In broadcast-Q mode dq is summed over all sequences.  Only valid
 * 128-key blocks of each (sequence, key/value head) are listed, sorted by cost
 * (see jfa_plan_bwd, called with num_kv_heads); they are taken in that order
 * under Cluster Launch Control, the default, or snake-dealt to one CTA per SM
 * under the static schedule (jfa_set_bwd_schedule).
 */
int jfa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
            void* dq, void* dk, void* dv, const int32_t* offsets_dev, const int32_t* offsets_host, int batch,
            int max_len, int nq_broadcast, int num_heads, int num_kv_heads, int head_dim, float scale, int causal,
            int broadcast_q, void* workspace, size_t workspace_bytes, void* stream);

/*
 * jfa_fwd_window, jfa_bwd_window -- jfa_fwd / jfa_bwd for self-attention under
 * a sliding window [C "performance and feature scope" and R "MXFP8 and
 * sparsity" name windows among the variants the kernels keep; the pages do not
 * define them, and this two-sided local window is this library's reading]:
 * query i of a sequence sees the keys j of its sequence with
 *   i - window_left <= j <= i + window_right,
 * where -1 leaves a side open.  (-1, -1) is jfa_fwd without causal masking,
 * (-1, 0) causal attention, (W-1, 0) causal attention over the last W keys.
 * Every query sees at least itself, so no output row is empty.  Each query
 * tile visits only the K/V blocks its rows can see (forward), and each key
 * block only the query tiles that see it (backward); blocks that straddle a
 * window edge are masked element-wise.  Bounds below -1 return
 * JFA_ERR_INVALID_ARG.  Other arguments, the workspace (jfa_workspace_size with
 * causal = 0) and lse as in jfa_fwd / jfa_bwd; the backward takes the lse of
 * the forward with the same window.
 */
int jfa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* offsets_dev,
                   const int32_t* offsets_host, int batch, int max_len, int num_heads, int num_kv_heads, int head_dim,
                   float scale, int window_left, int window_right, void* workspace, size_t workspace_bytes,
                   void* stream);
int jfa_bwd_window(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, const int32_t* offsets_dev, const int32_t* offsets_host, int batch,
                   int max_len, int num_heads, int num_kv_heads, int head_dim, float scale, int window_left,
                   int window_right, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Two-stage block-sparse forward [R "MXFP8 and sparsity": a cheap kernel
 * averages blocks of Q and K and picks the top-k most relevant key blocks,
 * then the attention kernel attends over those blocks only].  The pages give
 * neither block sizes, score nor tie rule; this library's reading: query
 * blocks of 256 rows (the forward's unit), key blocks of 128 keys, each
 * block's mean over the rows it really has, score = mean query . mean key
 * (key/value head h / (num_heads / num_kv_heads)), the topk highest scores,
 * ties to the lower block index, and exact softmax attention over every key of
 * the chosen blocks.  Self-attention or broadcast-Q, no causal mask.
 *
 * jfa_topk_rows: the number of query blocks (rows of the selection): for
 *   each sequence with keys, num_heads * ceil(rows / 256), rows = its length or
 *   nq_broadcast.  Returns the count or -jfa_status.
 * jfa_topk_select: first stage.  selection is device int32 [rows, topk], rows
 *   ordered by sequence, query head, query block; each row holds its chosen key
 *   block indices (0-based, within the sequence) in ascending order, then -1
 *   where the sequence has fewer than topk blocks.  Workspace:
 *   jfa_workspace_size(JFA_OP_TOPK_SELECT, ...).  Sequences of more than
 *   1,572,864 keys return JFA_ERR_UNSUPPORTED.
 * jfa_fwd_topk: second stage, o and lse as jfa_fwd, with the selection of
 *   jfa_topk_select (or any selection of ascending, in-range block indices,
 *   min(topk, blocks) of them per row).  Workspace:
 *   jfa_workspace_size(JFA_OP_FWD_TOPK, ...).
 */
int jfa_topk_rows(const int32_t* offsets_host, int batch, int nq_broadcast, int num_heads, int broadcast_q);
int jfa_topk_select(const void* q, const void* k, const int32_t* offsets_dev, const int32_t* offsets_host, int batch,
                    int max_len, int nq_broadcast, int num_heads, int num_kv_heads, int head_dim, int topk,
                    int broadcast_q, int32_t* selection, void* workspace, size_t workspace_bytes, void* stream);
int jfa_fwd_topk(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* selection,
                 int topk, const int32_t* offsets_dev, const int32_t* offsets_host, int batch, int max_len,
                 int nq_broadcast, int num_heads, int num_kv_heads, int head_dim, float scale, int broadcast_q,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * block_attn_fwd -- fixed 64-token block-diagonal self-attention [B 1, 2.1, 3].
 * Each sequence is cut into blocks of 64 tokens (the last one may be shorter)
 * and every block attends only within itself: one score GEMM and one PV GEMM per
 * block, no running-max correction, no log-sum-exp output.  num_kv_heads is
 * num_heads.  Programs get balanced contiguous ranges of (block pair, head)
 * tiles computed on the host in closed form [B 5].
 */
int block_attn_fwd(const void* q, const void* k, const void* v, void* o, const int32_t* offsets_dev,
                   const int32_t* offsets_host, int batch, int max_len, int num_heads, int head_dim, float scale,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * block_attn_bwd -- backward of block_attn_fwd [B 4]: P is recomputed from q and
 * k (no log-sum-exp tensor), Di is formed inline, and each block owns its own
 * dq, dk, dv rows, so no atomics are needed.  `o` is accepted for interface
 * symmetry; the kernel forms Di = rowsum(P o dP), which equals rowsum(dO o O).
 */
int block_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, void* dq,
                   void* dk, void* dv, const int32_t* offsets_dev, const int32_t* offsets_host, int batch,
                   int max_len, int num_heads, int head_dim, float scale, void* workspace, size_t workspace_bytes,
                   void* stream);

/*
 * block_attn_fwd_rope, block_attn_bwd_rope -- block_attn_fwd / block_attn_bwd
 * with a rotary position embedding of q and k fused into the kernels [B
 * introduction: "with rotary fused"].  The pages do not state the rotary
 * convention; this library's reading is the rotate-half form: the position of
 * a row is its index inside its sequence, and for i < head_dim/2 the pair
 * (x_i, x_{i+head_dim/2}) of a q or k row at position p turns by the angle
 * a(p, i):
 *   (x_i, x_{i+D/2}) -> (x_i cos a - x_{i+D/2} sin a, x_{i+D/2} cos a + x_i sin a).
 * rope_cos and rope_sin are fp32 device tables [rope_rows, head_dim/2] (row p,
 * column i = cos / sin of a(p, i); any angles, e.g. p * base^(-2i/D)), 16-byte
 * aligned, rope_rows >= max_len.  The forward attends with the rotated q and k;
 * the backward recomputes them and returns dq and dk with respect to the
 * unrotated q and k (the transposed rotation is applied before they are
 * returned).  q and k stay unrotated in memory: the kernels rotate their tiles
 * in shared memory, from the tables packed into the workspace as fp16 words
 * (for each two column pairs, one word of their cosines and one of their
 * sines), whose size is jfa_workspace_size(JFA_OP_BLOCK_FWD_ROPE or
 * JFA_OP_BLOCK_BWD_ROPE, ...) (the plain size plus longest sequence x
 * head_dim/2 x 4 bytes); the backward kernel's epilogue carries dq and dk
 * back through the transposed rotation before it stores them.  Errors as
 * block_attn_*, plus JFA_ERR_INVALID_ARG for missing, misaligned or too short
 * tables.
 */
int block_attn_fwd_rope(const void* q, const void* k, const void* v, void* o, const float* rope_cos,
                        const float* rope_sin, int rope_rows, const int32_t* offsets_dev,
                        const int32_t* offsets_host, int batch, int max_len, int num_heads, int head_dim,
                        float scale, void* workspace, size_t workspace_bytes, void* stream);
int block_attn_bwd_rope(const void* q, const void* k, const void* v, const void* o, const void* dout, void* dq,
                        void* dk, void* dv, const float* rope_cos, const float* rope_sin, int rope_rows,
                        const int32_t* offsets_dev, const int32_t* offsets_host, int batch, int max_len,
                        int num_heads, int head_dim, float scale, void* workspace, size_t workspace_bytes,
                        void* stream);

/*
 * jfa_fwd_noalloc -- jfa_fwd for callers that cannot allocate device memory.
 * The pages have no counterpart of this entry point.  Some callers cannot give
 * the library a workspace: code inside a host framework whose memory manager
 * owns all device memory and forbids extensions from calling cudaMalloc, or a
 * serving loop that must never allocate.  This variant takes the same arguments
 * as jfa_fwd minus the workspace and keeps its scratch (tile plan, error word,
 * empty-sequence list) in one static device array of jfa_fwd_noalloc_capacity()
 * bytes (1 MiB), held by every GPU that loads the library until the process
 * exits.  A problem whose plan does not fit returns JFA_ERR_TOO_LARGE (about
 * 60,000 forward units of 256 query rows).  It calls no cudaMalloc, cudaFree or
 * other allocating routine.  All calls share the array: calls that overlap on
 * the GPU (different streams with no ordering) race, and the array keeps the
 * last call's contents (each call clears the error word first).  The first call
 * on each device looks up the array's device address; make it before any
 * stream capture.  The plan is copied from pageable host memory, so each call
 * returns only once the work already queued on `stream` has finished.
 */
int jfa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, const int32_t* offsets_dev,
                    const int32_t* offsets_host, int batch, int max_len, int nq_broadcast, int num_heads,
                    int num_kv_heads, int head_dim, float scale, int causal, int broadcast_q, void* stream);
/* Size in bytes of jfa_fwd_noalloc's static scratch array. */
size_t jfa_fwd_noalloc_capacity(void);
/*
 * jfa_fwd_noalloc_status -- the counterpart of jfa_device_status for
 * jfa_fwd_noalloc: synchronises `stream` and returns JFA_OK, or
 * JFA_ERR_DEVICE_TIMEOUT if a kernel recorded a failure (a bounded wait that
 * ran out) in the static array's error word since the last jfa_fwd_noalloc
 * call on the current device.  Allocates nothing.
 */
int jfa_fwd_noalloc_status(void* stream);
/*
 * jfa_selftest_wait_timeout_noalloc -- the failure-path self-test (see
 * jfa_selftest_wait_timeout) with its error word in jfa_fwd_noalloc's static
 * array: after about 2 s jfa_fwd_noalloc_status() reports
 * JFA_ERR_DEVICE_TIMEOUT; the next jfa_fwd_noalloc call clears it.
 */
int jfa_selftest_wait_timeout_noalloc(void* stream);

/*
 * jfa_workspace_size -- device workspace in bytes that `op` needs for this
 * problem (plans, per-row Di, the fp32 dQ accumulator, an error word).
 * Returns 0 on invalid arguments.  Queries the current device's SM count.
 * num_heads is the number of query heads; for a GQA backward the size is an
 * upper bound (the call plans over the fewer key/value heads).
 */
size_t jfa_workspace_size(int op, const int32_t* offsets_host, int batch, int nq_broadcast, int num_heads,
                          int head_dim, int causal, int broadcast_q);

/* Human-readable name of a jfa_status value (static string). */
const char* jfa_status_string(int status);

/*
 * jfa_device_status -- synchronises `stream` and returns JFA_OK or the error a
 * kernel recorded in `workspace` since the last call that used it.
 */
int jfa_device_status(const void* workspace, void* stream);

/*
 * Host planners, exported so tests can compare them bit for bit with a naive
 * restatement [R "Tile balancing and Cluster Launch Control"; B 5].
 * Entries are int32 quadruples (b, h, tile, cost), CTA-major, with cta_start
 * [n_cta+1] giving each CTA's slice.  Pass NULL buffers to only count.
 * Return the number of units (>= 0) or -jfa_status.
 *
 *   jfa_plan_fwd: unit = 256 query rows (b, h, m); cost = 128-key blocks
 *     visited; stable sort by cost descending; snake deal over n_cta.
 *   jfa_plan_bwd: unit = one valid 128-key block (b, h, n), enumerated b, h, n
 *     (n innermost); cost = 128-row query tiles visited per query head; stable
 *     sort by cost descending, snake deal (equal costs keep the enumeration
 *     order).  h runs over the key/value heads: jfa_bwd passes num_kv_heads
 *     here, and each unit then visits the tiles of its G query heads.
 */
int jfa_plan_fwd(const int32_t* offsets_host, int batch, int num_heads, int nq_broadcast, int causal, int n_cta,
                 int32_t* units, int32_t* cta_start);
int jfa_plan_bwd(const int32_t* offsets_host, int batch, int num_heads, int nq_broadcast, int causal, int n_cta,
                 int32_t* units, int32_t* cta_start);
/*
 *   jfa_plan_window: the same planners for self-attention under a window (see
 *     jfa_fwd_window): which = 0 forward (as jfa_plan_fwd), 1 backward (as
 *     jfa_plan_bwd).  A unit's cost counts the blocks or tiles it visits
 *     inside the window.
 */
int jfa_plan_window(int which, const int32_t* offsets_host, int batch, int num_heads, int window_left,
                    int window_right, int n_cta, int32_t* units, int32_t* cta_start);
/*
 *   block_plan: block_per_batch [batch+1] = exclusive prefix sum of ceil(L/64);
 *     tiles are pairs of consecutive global blocks per head (id = pair*H + h);
 *     prog_start [P+1] with P = min(n_sm, tiles) from closed-form divmod.
 *     Either buffer may be NULL.  Returns P (>= 0) or -jfa_status.
 */
int block_plan(const int32_t* offsets_host, int batch, int num_heads, int n_sm, int32_t* block_per_batch,
               int32_t* prog_start);

/*
 * Work distribution of the persistent jagged forward [R "Tile balancing and
 * Cluster Launch Control"; C "load balancing"].
 *   0  static plan: units sorted by cost and snake-dealt to one CTA per SM;
 *   1  Cluster Launch Control: one CTA per unit, launched in cost order; a CTA
 *      that finishes a unit cancels the launch of a CTA that has not started
 *      yet and processes that CTA's unit instead, so residual imbalance is
 *      absorbed at run time.
 * The initial mode comes from the environment variable JFA_SCHED ("static" or
 * "clc"), else the library default; jfa_set_schedule() changes it for
 * subsequent calls (process-wide).  jfa_get_schedule() returns the mode in use.
 */
int jfa_set_schedule(int mode);
int jfa_get_schedule(void);

/*
 * The same two modes for the jagged backward's persistent kernel, whose units
 * are 128-key blocks [R "Tile balancing and Cluster Launch Control"]: 0 static
 * plan (units sorted by cost, snake-dealt over one CTA per SM), 1 Cluster Launch
 * Control (one CTA per unit in cost order; a CTA that finishes a unit takes
 * over the unit of a CTA not yet launched).  Initially JFA_SCHED_BWD ("static"
 * or "clc") if set, else Cluster Launch Control; jfa_set_bwd_schedule() changes it for
 * subsequent calls (process-wide).  Returns JFA_ERR_INVALID_ARG for another mode.
 */
int jfa_set_bwd_schedule(int mode);
int jfa_get_bwd_schedule(void);

/*
 * The same two modes for the block-diagonal kernels [B 5; R "Tile balancing and
 * Cluster Launch Control"]: 0 closed-form static ranges (programs get balanced
 * contiguous ranges of (block pair, head) tiles, one CTA per SM); 1 Cluster
 * Launch Control (one CTA per chunk of 16 consecutive tiles; a CTA that
 * finishes a chunk takes over the chunk of a CTA not yet launched).  Both
 * modes give bit-identical results (every tile owns its outputs).  Initially
 * JFA_SCHED_BLOCK ("static" or "clc") if set, else Cluster Launch Control;
 * jfa_set_block_schedule() changes it for subsequent calls (process-wide).
 */
int jfa_set_block_schedule(int mode);
int jfa_get_block_schedule(void);

/*
 * Optional kernel timing (no counterpart on the pages; measurement support).
 * jfa_profile_enable(1) starts counting every library kernel launch and
 * bracketing it with CUDA events on its stream (and forgets earlier records);
 * jfa_profile_enable(0) stops it.  jfa_profile_select(mask) limits the events
 * to the kinds whose bit is set in mask (launches of the other kinds are still
 * counted; the initial mask selects every kind; a mask outside [0, 2^9)
 * returns JFA_ERR_INVALID_ARG), so a measurement can time one kernel without
 * adding events around the rest.  jfa_profile_read(kind, &ms, &n) synchronises
 * on the recorded events and returns the summed device time (0 for an
 * unselected kind) and the launch count of one kernel kind: 0 forward,
 * 1 backward prepass (Di), 2 backward main, 3 dQ convert, 4 block forward,
 * 5 block backward, 6 empty-sequence fill, 7 top-k selection, 8 rotary table
 * packing.
 */
/*
 * Failure-path self-test (no counterpart on the pages; failure detection).
 * Launches on `stream` one CTA that waits, through the same bounded mbarrier
 * wait every kernel of this library uses, on a barrier that nothing completes.
 * The wait gives up after its limit (2 s), the CTA records
 * JFA_ERR_DEVICE_TIMEOUT in the error word at the start of `workspace` (device
 * memory, at least 4 bytes, owned by the caller) and exits; no fault, no trap,
 * and the context stays usable.  Returns JFA_ERR_INVALID_ARG for a null or too
 * small workspace, JFA_ERR_CUDA if the launch fails, else JFA_OK; read the
 * outcome with jfa_device_status(workspace, stream).
 */
int jfa_selftest_wait_timeout(void* workspace, size_t workspace_bytes, void* stream);

int jfa_profile_enable(int on);
int jfa_profile_select(int kind_mask);
int jfa_profile_read(int kind, double* total_ms, int* launches);

#ifdef __cplusplus
}
#endif
#endif /* JFA_H_ */
