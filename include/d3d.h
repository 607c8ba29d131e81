/*
 * d3d.h — C ABI of the GB300 (sm_103a) hot path of diffusion-drafted
 * speculative decoding: packed drafting attention, speculative-sampling
 * verification, and the branch cache-hit match.
 *
 * Sources:
 *   [D3D]    "D3D: Decoupled Diffusion Drafting for Asynchronous Speculative
 *            Decoding" (paper summary page and arXiv abstract).
 *   [DScout] "Factorization-Guided Training and Inference for
 *            Diffusion-Drafted Speculative Decoding" (paper summary page).
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers to caller-owned memory, unless an
 *     argument says "host".  The library never allocates device memory,
 *     keeps no state between calls, and never frees anything.
 *   - Work is enqueued on `stream`; the call returns once it is enqueued.
 *     Outputs are valid after the stream reaches that point.
 *   - Return value: D3D_OK, or a negative D3D_ERR_* code, in which case
 *     nothing was enqueued.  Problems that can only be seen on the device
 *     (a descriptor that lies, a bounded wait that expired) are recorded in
 *     the status word at the start of the call's workspace; read it with
 *     d3d_workspace_status().  Kernels never trap.
 *   - Scratch ("workspace") is caller-allocated device memory of at least
 *     the size the matching *_workspace_size() function returns, 256-byte
 *     aligned, zero-filled once before its first use (d3d_workspace_init),
 *     and not written by the caller between calls.  The kernels leave it
 *     ready for the next call.  Calls that share one workspace must be
 *     ordered on the device (same stream, or events).
 *   - Layouts are row-major and dense (innermost dimension contiguous).
 *     bf16 is IEEE bfloat16 stored as 16-bit words.
 */
#ifndef D3D_H_
#define D3D_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define D3D_OK 0
#define D3D_ERR_INVALID_ARG (-1)     /* a host-visible argument is invalid            */
#define D3D_ERR_UNSUPPORTED (-2)     /* valid but not implemented (e.g. head_dim)    */
#define D3D_ERR_WORKSPACE (-3)       /* workspace NULL, misaligned or too small      */
#define D3D_ERR_CUDA (-4)            /* a CUDA runtime call failed at enqueue time   */
#define D3D_ERR_DEVICE_TIMEOUT (-5)  /* device status: a bounded wait expired        */
#define D3D_ERR_DEVICE_INPUT (-6)    /* device status: device-side data out of range */
#define D3D_ERR_INTERNAL (-7)        /* device status, debug build only: an internal
                                        index check failed (the access was skipped)  */

/* ---- enums -------------------------------------------------------------- */
#define D3D_DTYPE_F32 0
#define D3D_DTYPE_BF16 1

#define D3D_SEG_CAUSAL 0 /* token i of the segment sees tokens 0..i of it      */
#define D3D_SEG_BIDIR 1  /* every token of the segment sees the whole segment  */

/*
 * One segment of a request's packed query sequence ([D3D] "Background:
 * asynchronous drafting and cache hits" and "Method steps", step 4: one
 * packed forward drafts successor blocks for every rejection position and
 * alternative anchor, plus the all-accept case).  Fields are local to the
 * request: q_start is the first packed token of the segment, len its token
 * count (>= 1); parent is the index (within the request) of an earlier
 * causal segment without a parent whose first parent_len tokens this
 * segment also sees, or -1 (then parent_len = 0).  Segments tile the
 * request's packed tokens in order.
 */
typedef struct {
    int32_t q_start;
    int32_t len;
    int32_t mode;
    int32_t parent;
    int32_t parent_len;
} d3d_segment_t;

/* Text for a status code (static storage; never NULL). */
const char *d3d_status_string(int status);

/* Library version as 10000*major + 100*minor + patch. */
int d3d_version(void);

/* Zero `bytes` of workspace on `stream` (first use, or after a device error). */
int d3d_workspace_init(void *ws, size_t bytes, cudaStream_t stream);

/* Copy the workspace status word to *status_host (synchronises `stream`) and,
 * if `clear` is nonzero, reset it to D3D_OK.  Returns D3D_OK or D3D_ERR_CUDA. */
int d3d_workspace_status(const void *ws, int32_t *status_host, int clear, cudaStream_t stream);

/*
 * Host-side check of a segment table (all pointers HOST): segments tile
 * each request in order with no gap or overlap, len >= 1, mode is causal or
 * bidirectional, a parent is an earlier causal segment of the same request
 * with no parent of its own (one nesting level), 0 <= parent_len <=
 * len(parent), parent_len = 0 without a parent, cu_q/cu_seg start at 0 and
 * do not decrease.  Returns D3D_OK or D3D_ERR_INVALID_ARG.
 */
int d3d_validate_segments(const d3d_segment_t *segs, const int32_t *cu_q, const int32_t *cu_seg, int R);

/* ========================================================================
 * Packed drafting attention.
 *
 * [D3D] "Core method" and "Method steps" (steps 2 and 4): every draft block
 * (anchor + mask tokens) attends to the shared prefix, causally to the
 * hypothesised accepted tokens of its branch, and bidirectionally within
 * itself; one packed pass covers N_async = B[(C-1)F+2] query tokens.
 * [DScout] "Background: block-diffusion drafter": one forward predicts all
 * mask positions of a block of the latest target token plus bs-1 masks.
 *
 * For request r, packed query token i (local) and query head h, with
 * G = Hq/Hkv and kv head h/G:
 *   out[i,h] = sum_k softmax_k(scale * <q[i,h], K[k]>) V[k]
 * over the visible keys k: all prefix rows cu_prefix[r] .. cu_prefix[r+1]-1
 * of k_prefix/v_prefix, and the packed rows j of k_packed/v_packed (rows
 * cu_q[r] + j) that are in i's own segment (j <= i when causal) or among
 * the first parent_len tokens of its parent segment.
 *
 *   q           [total_q, Hq, d] bf16      query rows (RoPE already applied)
 *   k_prefix    [total_prefix, Hkv, d] bf16 cached keys of the shared prefix
 *   v_prefix    [total_prefix, Hkv, d] bf16
 *   k_packed    [total_q, Hkv, d] bf16     keys/values of the packed tokens
 *   v_packed    [total_q, Hkv, d] bf16
 *   segs        [total_segs] d3d_segment_t (device)
 *   cu_prefix   [R+1] int32 (device) prefix row offsets, cu_prefix[0] = 0,
 *               cu_prefix[R] = total_prefix
 *   cu_q        [R+1] int32 (device) packed row offsets, cu_q[0] = 0, cu_q[R] = total_q
 *   cu_seg      [R+1] int32 (device) segment offsets, cu_seg[0] = 0,
 *               cu_seg[R] = total_segs.  With R == 1 these fix every offset,
 *               so the kernel starts from the totals and checks the arrays
 *               against them afterwards (a mismatch: D3D_ERR_DEVICE_INPUT in
 *               the status word and a zero output)
 *   max_q, max_prefix  host upper bounds of any request's packed / prefix
 *               length (they size the grid; a request beyond them is a
 *               device input error); max_q <= 8192 (64 tiles of 128 rows,
 *               else D3D_ERR_UNSUPPORTED)
 *   q, k_*, v_*, out  16-byte aligned (the tensor maps' base rule; else
 *               D3D_ERR_INVALID_ARG)
 *   d           64 or 128 (else D3D_ERR_UNSUPPORTED); Hq % Hkv == 0 and
 *               128 % (Hq/Hkv) == 0
 *   scale       softmax scale (normally 1/sqrt(d))
 *   out         [total_q, Hq, d] bf16
 *   ws          workspace, d3d_packed_draft_attn_workspace_size() bytes (the
 *               status word only: the key splits of a query tile combine
 *               their partial results through distributed shared memory of
 *               a thread-block cluster, not through global scratch)
 *   max_ctas    0: the plan may use every SM.  n > 0: a budget of n SMs
 *               (each CTA holds one), so that a kernel running beside the
 *               attention keeps the others: the plan picks its kernel and key
 *               split for a wave of at most n CTAs.  The launch never has
 *               fewer CTAs than the unsplit plan (one per query-tile pair of
 *               each request and KV head, R * Hkv * ceil(MT / 2), MT the
 *               query tiles of a head group): a budget below that count is
 *               exceeded (the CTAs then run in more than one wave when they
 *               outnumber the free SMs).  Results do not depend on it.  Negative:
 *               D3D_ERR_INVALID_ARG.
 *   flags       0, or D3D_ATTN_AFTER_INDEPENDENT: the launch may start while
 *               the kernel before it on the stream still runs (programmatic
 *               dependent launch) -- for the verification of the same round,
 *               launched first with an sm_limit, whose output the attention
 *               does not read.  The attention still finishes only after that
 *               kernel has finished, so later work on the stream sees both.
 *               Or D3D_ATTN_AFTER_DEPENDENT: the launch may also start while
 *               the kernel before it runs, but it waits for that kernel to
 *               finish (and its writes to be visible) before it reads any
 *               input; only its setup (barriers, TMEM, tensor-map prefetch)
 *               overlaps -- for the next round's attention after this round's
 *               kernels.  The two bits are exclusive.  Other bits:
 *               D3D_ERR_INVALID_ARG.
 * Device-side checks: offsets out of the totals' range or a segment table
 * that breaks the rules of d3d_validate_segments set D3D_ERR_DEVICE_INPUT
 * in the status word (the affected rows are written as zeros).
 * The launch holds one or two 128-row query tiles per CTA (two halve the K/V
 * bytes each SM receives per flop) and splits the keys of a tile (pair) over
 * up to 8 CTAs of a cluster; the plan minimises the estimated time on the
 * device's SMs (or max_ctas of them).
 * ======================================================================== */
#define D3D_ATTN_AFTER_INDEPENDENT 1
#define D3D_ATTN_AFTER_DEPENDENT 2

size_t d3d_packed_draft_attn_workspace_size(int R, int Hq, int Hkv, int d, int max_q, int max_prefix);

/* Number of CTAs the d3d_packed_draft_attn launch for these sizes (and this
 * max_ctas) uses on the current device; each holds one SM from its start to
 * its end (they all fit in one wave when the count is at most the SM count).  A caller that runs
 * another kernel beside the attention can give it the remaining SMs (see
 * d3d_spec_verify's sm_limit).  Returns the count, or a negative status for
 * arguments d3d_packed_draft_attn would reject (D3D_ERR_INVALID_ARG,
 * D3D_ERR_UNSUPPORTED); 0 when there is nothing to compute. */
int d3d_packed_draft_attn_ctas(int R, int Hq, int Hkv, int d, int max_q, int max_prefix, int max_ctas);

int d3d_packed_draft_attn(const void *q, const void *k_prefix, const void *v_prefix, const void *k_packed,
                          const void *v_packed, const d3d_segment_t *segs, const int32_t *cu_prefix,
                          const int32_t *cu_q, const int32_t *cu_seg, int R, int Hq, int Hkv, int d,
                          int max_q, int max_prefix, int total_q, int total_prefix, int total_segs,
                          float scale, void *out, void *ws, size_t ws_bytes, int max_ctas, int flags,
                          cudaStream_t stream);

/*
 * Failure-detection hook (no counterpart on the pages).  mode 1 makes every
 * later d3d_packed_draft_attn launch skip its first key-tile load, so the
 * consumer's bounded wait expires: the kernel records D3D_ERR_DEVICE_TIMEOUT
 * in the workspace status word, releases its resources and returns.  mode 2
 * makes every later d3d_spec_verify launch that copies logit rows into
 * shared memory by bulk copies skip one copy of CTA 0: its first item's
 * copies in the ring of an sm_limit launch over bf16 rows, or its first row
 * in the vocabulary-slice launch.  That CTA's bounded wait expires, it
 * records D3D_ERR_DEVICE_TIMEOUT, waits out its other copies and leaves, and
 * the request's other CTAs give up their bounded waits.  The outputs of such a call are undefined and the
 * workspace must be re-initialised.  mode 0 (the default) restores normal
 * operation.  The setting is process-global and not thread-safe.
 */
void d3d_debug_inject_fault(int mode);

/*
 * Kernel selection hook for tests and measurements (no counterpart on the
 * pages).  d3d_packed_draft_attn and d3d_packed_draft_attn_ctas plan their
 * launch among three kernels of equal results: 1 one query tile per CTA
 * (with key splits), 2 two query tiles per CTA (with key splits), 3 CTA
 * pairs sharing their MMAs (one tile per CTA, head_dim 128 only, no key
 * splits).  kind 1..3 restricts later plans to that kernel where it applies
 * (elsewhere the plan chooses as usual); 0 (the default) lets the plan
 * choose.  Other values: ignored.  The setting is process-global and not
 * thread-safe.
 */
void d3d_debug_force_attn_kernel(int kind);

/* ========================================================================
 * Acceptance probabilities and expected acceptance length.
 *
 * [DScout] "Background: AWL and the acceptance rule": position j accepts its
 * draft token with probability a_j = sum_v min(P_j(v), Q_j(v));
 * [DScout] "Background: acceptance length tau": the prefix survival
 * S(k) = a_1 ... a_k and tau = 1 + sum_{k=1}^{B-1} S(k).  P_j and Q_j as in
 * d3d_spec_verify (softmax of the target and draft rows at temperature T).
 *
 *   target_logits [R, B, V], draft_logits [R, B-1, V] f32 or bf16 (row B-1 of
 *               the target is not read)
 *   temperature > 0 (else D3D_ERR_INVALID_ARG)
 *   accept_prob [R, B-1] float32 output; survival [R, B-1] and tau [R]
 *               float32 outputs, each may be NULL
 *   ws          d3d_accept_probs_workspace_size() bytes (enough for either
 *               shape; a smaller one that still holds the two launches'
 *               chunk records makes the call take that shape)
 * When each request's rows split over the device's SMs with the 2(B-1) rows
 * of a vocabulary slice resident in one CTA's shared memory: one cooperative
 * launch, one CTA per (request, slice), the logits read once.  Otherwise two
 * launches on the stream (the second a programmatic dependent of the first),
 * the logits read twice.  fp32 arithmetic, sums in a fixed order (results do
 * not depend on scheduling); a_j is clamped to 1.  2 <= B <= 257 (B > 257:
 * D3D_ERR_UNSUPPORTED).
 * ======================================================================== */
size_t d3d_accept_probs_workspace_size(int R, int B, int V);

int d3d_accept_probs(const void *target_logits, const void *draft_logits, int logits_dtype, int R, int B, int V,
                     float temperature, float *accept_prob, float *survival, float *tau, void *ws, size_t ws_bytes,
                     cudaStream_t stream);

/* ========================================================================
 * Branch construction for the asynchronous packed pass.
 *
 * [D3D] "Background: asynchronous drafting and cache hits", "Method steps"
 * (step 4): the packed pass drafts, for every rejection position, one block
 * from each of F alternative anchors, plus the all-accept block.  This call
 * builds that pass's segment rows and the branches' heads (the inputs of
 * d3d_packed_draft_attn and of the branch match) from the drafter's logits.
 * Reading (the pages do not say how anchors are chosen): the anchors of
 * rejection position p (0-based draft index, p = 0..C-2) are the F tokens
 * with the largest draft logit in row p (ties to the lowest index), the
 * drafted token y_p excluded.
 *
 * With M = (C-1)F + 2 branches per request, indexed like the segments:
 *   anchors  [R, C-1, F] int32 (may be NULL when (C-1)F == 0)
 *   heads    [R, M, B] int32: branch 0 (the block under verification) is
 *            empty; branch k = 1 + pF + f is y_0 .. y_{p-1}, anchor (p, f);
 *            branch M-1 is y_0 .. y_{B-2}, bonus_guess[r]; entries past the
 *            length are -1
 *   head_len [R, M] int32: 0, p + 1, and B (0 when bonus_guess is NULL:
 *            without a guess of the bonus token that branch never matches)
 *   segs     [R*M] d3d_segment_t, request-local rows (may be NULL):
 *            (0, B, causal, -1, 0), (kB, B, bidirectional, 0, p+1),
 *            ((M-1)B, B, bidirectional, 0, B)
 *   cu_q, cu_seg [R+1] int32: r*M*B and r*M (both NULL or both given)
 *   draft_logits [R, B-1, V] f32 or bf16; draft_tokens [R, B-1] int32;
 *   bonus_guess [R] int32 or NULL
 *   ws       d3d_build_branches_workspace_size() bytes
 * 1 <= C <= B, F >= 0, F <= V-1 when there are anchors (else
 * D3D_ERR_INVALID_ARG); B <= 256, F <= 8, (C-1)F <= 256 and R*M*B < 2^31
 * (else D3D_ERR_UNSUPPORTED).  A draft token outside [0, V) sets
 * D3D_ERR_DEVICE_INPUT (nothing is excluded in its row).  No CTA of the
 * launch waits for another.
 * ======================================================================== */
size_t d3d_build_branches_workspace_size(int R, int B, int V, int C, int F);

int d3d_build_branches(const void *draft_logits, int logits_dtype, const int32_t *draft_tokens,
                       const int32_t *bonus_guess, int R, int B, int V, int C, int F, int32_t *anchors,
                       int32_t *heads, int32_t *head_len, d3d_segment_t *segs, int32_t *cu_q, int32_t *cu_seg,
                       void *ws, size_t ws_bytes, cudaStream_t stream);

/* ========================================================================
 * Speculative-sampling verification.
 *
 * [D3D] "Background: speculative decoding": accept the drafted prefix by
 * rejection sampling and resample one token from the residual distribution
 * at the first rejection, so the output follows the target exactly.
 * [DScout] "Background: speculative decoding": accept the prefix before the
 * first rejected token, add a replacement there, or a bonus token when all
 * drafts are accepted.  [DScout] "Background: AWL and the acceptance rule":
 * alpha_j = min(1, P_j(y_j) / Q_j(y_j)).
 *
 * Per request r (0-based rows: target row j is P_{j+1}, row B-1 is P_B):
 *   P_j = softmax(target[r,j,:] / T), Q_j = softmax(draft[r,j,:] / T)
 *   alpha_j = min(1, P_j(y_j) / Q_j(y_j))          (1 when Q_j(y_j) <= P_j(y_j))
 *   a = number of leading j with u_accept[r,j] < alpha_j
 *   if a < B-1: t = InvCDF(max(0, P_a - Q_a), u_sample[r])   (row a = P_{a+1})
 *              (if that residual sums to 0 in fp32: InvCDF(P_a, u_sample[r]))
 *   else:       t = InvCDF(P_{B-1}, u_sample[r])               (bonus, P_B)
 *   InvCDF(w, u) = smallest v (ascending) with sum_{x<=v} w_x > u * sum(w)
 *   out_tokens[r] = [y_0 .. y_{a-1}, t, -1, ...], num_tokens[r] = a + 1
 *   (the round's tau: accepted drafts plus the target's own token).
 *
 * Launch shapes (results do not depend on them): when every request's rows
 * split over the SMs the launch may use (sm_limit, else the device) with
 * the 2B-1 rows of each vocabulary slice resident in one CTA's shared
 * memory, each CTA holds one (request, slice) and reads its rows once;
 * otherwise CTAs take (request, position, chunk) items and reload the
 * sampled row.  Both wait on one another through the workspace.
 *
 * Greedy verification, temperature == 0 ([D3D] "Experiments", [DScout]
 * "Experiments": the pages' results are greedy; the T -> 0 limit of the
 * rule above).  g_j = argmax_v target[r,j,v], ties to the lowest index;
 *   a = number of leading j with y_j == g_j,  t = g_a  (g_{B-1}: the bonus);
 *   alpha_j = p_draft_j = 1 if y_j == g_j else 0.
 * Only the target logits are read: draft_logits, u_accept and u_sample may
 * be NULL, q_draft must be NULL (else D3D_ERR_INVALID_ARG).  The launch
 * needs no co-residency: every CTA finishes its part without waiting.
 *
 *   target_logits [R, B, V], draft_logits [R, B-1, V]  f32 or bf16 (logits_dtype)
 *   draft_tokens  [R, B-1] int32 in [0, V)
 *   u_accept [R, B-1], u_sample [R]  float32 in [0, 1)
 *   temperature   > 0 (sampling) or 0 (greedy); negative or not finite:
 *               D3D_ERR_INVALID_ARG
 *   B >= 2, V >= 1 (else D3D_ERR_INVALID_ARG); B > 256 or V > 8388608
 *               (1024 chunks of 8192 logits): D3D_ERR_UNSUPPORTED
 *   accept_len [R], out_tokens [R, B], num_tokens [R]  int32 outputs
 *   alpha, p_draft, q_draft [R, B-1] float32 outputs, each may be NULL
 *               (p_draft = P_j(y_j), q_draft = Q_j(y_j))
 *   awl_weight  [R, B-1] float32 output or NULL: the acceptance-weighted loss
 *               weight of [DScout] "Background: AWL and the acceptance rule",
 *               w_k = prod_{j<k} alpha_j (w_0 = 1), the probability that
 *               verification reaches position k given the drafted tokens; a
 *               running fp32 product in position order (greedy: the product
 *               of the acceptance indicators)
 *   heads [R, M, B], head_len [R, M], branch [R]  int32; optional fused
 *               branch match: when branch is not NULL, the kernel writes
 *               branch[r] exactly as d3d_branch_match would for the verified
 *               tokens out_tokens[r, :num_tokens[r]] (heads/head_len may be
 *               NULL when M == 0).  The heads are the round's inputs ([D3D]
 *               "Background: asynchronous drafting and cache hits": each
 *               branch hypothesises an accepted prefix and its corrected
 *               token), so the match needs nothing from the drafting pass.
 *   ws          workspace, d3d_spec_verify_workspace_size() bytes (enough
 *               for every launch shape; a smaller one that still holds the
 *               chunked launch's records makes the call take that shape)
 *   sm_limit    0: the kernel may use every SM.  n > 0: at most n CTAs, each
 *               holding a whole SM, so that a kernel running beside it (the
 *               drafting attention of the same round, launched as its
 *               programmatic dependent or on another stream) keeps the
 *               remaining SMs whichever starts first.  Results do not depend
 *               on it.  Negative: D3D_ERR_INVALID_ARG.
 *   flags       0, or D3D_VERIFY_AFTER_INDEPENDENT: the launch may start
 *               while the kernel before it on the stream still runs
 *               (programmatic dependent launch) -- for the drafting attention
 *               of the same round, launched first, whose output the
 *               verification does not read; give an sm_limit that leaves the
 *               attention's SMs.  The verification still finishes only after
 *               that kernel has finished.  Other bits: D3D_ERR_INVALID_ARG.
 * A draft token outside [0, V) sets D3D_ERR_DEVICE_INPUT in the status word
 * and is treated as rejected (alpha = 0).
 * ======================================================================== */
#define D3D_VERIFY_AFTER_INDEPENDENT 1

size_t d3d_spec_verify_workspace_size(int R, int B, int V);

/* Launch shape of d3d_spec_verify for these sizes on the current device,
 * with 16-byte aligned logit pointers and a workspace of ws_bytes: the
 * number of CTAs of the vocabulary-slice launch (R times the slices of a
 * request; each holds one SM from its start to its end), or 0 when the call
 * takes the chunked launch (or the greedy one, temperature == 0, or R == 0).
 * D3D_ERR_INVALID_ARG for sizes d3d_spec_verify would reject. */
int d3d_spec_verify_slice_ctas(int R, int B, int V, int logits_dtype, float temperature, int sm_limit,
                               size_t ws_bytes);

int d3d_spec_verify(const void *target_logits, const void *draft_logits, int logits_dtype,
                    const int32_t *draft_tokens, const float *u_accept, const float *u_sample, int R, int B,
                    int V, float temperature, int32_t *accept_len, int32_t *out_tokens, int32_t *num_tokens,
                    float *alpha, float *p_draft, float *q_draft, float *awl_weight, const int32_t *heads,
                    const int32_t *head_len, int M, int32_t *branch, void *ws, size_t ws_bytes, int sm_limit,
                    int flags, cudaStream_t stream);

/*
 * Verification that allocates nothing (the pages have no counterpart: this
 * is a calling convenience of this library).
 *
 * Some callers cannot allocate device memory at all: a serving process whose
 * memory manager has already reserved the whole GPU for model weights and KV
 * cache, code in a latency-critical loop that cannot afford the device-wide
 * synchronisation cudaMalloc implies, or a caller behind a C interface with
 * no allocator to hand.  This entry point computes exactly what
 * d3d_spec_verify computes, with the same arguments minus the workspace; its
 * scratch is a fixed 2 MiB array inside the library, which every device that
 * loads the library holds until the process exits.
 *
 *   - Problems whose d3d_spec_verify_workspace_size(R, B, V) exceeds 2 MiB
 *     are rejected with D3D_ERR_UNSUPPORTED (for B = 16 and V = 151936 the
 *     largest accepted batch is R = 211 requests); use d3d_spec_verify for
 *     larger ones.
 *   - The first call on each device looks up the array's device address with
 *     that device current and keeps it for the life of the process; make that
 *     first call before any stream capture.  cudaDeviceReset (or any teardown
 *     of the device's primary context) invalidates the kept address: do not
 *     call this entry point on a device after resetting it.
 *   - Every call shares the one array per device: calls that overlap on the
 *     GPU (different streams without ordering between them) race and give
 *     wrong results.  Each call zeroes the parts that must start at zero.
 *   - The status word of this entry point lives inside the fixed array and
 *     is not reported back: a draft token outside [0, V) is handled as in
 *     d3d_spec_verify, and a device-side wait that expires (see
 *     D3D_ERR_DEVICE_TIMEOUT) leaves the outputs undefined, yet the call
 *     still returns D3D_OK.  Call d3d_spec_verify when that status is needed.
 * Returns D3D_OK, D3D_ERR_INVALID_ARG, D3D_ERR_UNSUPPORTED or D3D_ERR_CUDA.
 */
int d3d_spec_verify_noalloc(const void *target_logits, const void *draft_logits, int logits_dtype,
                            const int32_t *draft_tokens, const float *u_accept, const float *u_sample, int R, int B,
                            int V, float temperature, int32_t *accept_len, int32_t *out_tokens, int32_t *num_tokens,
                            float *alpha, float *p_draft, float *q_draft, cudaStream_t stream);

/* ========================================================================
 * The asynchronous round in one launch.
 *
 * [D3D] "Background: asynchronous drafting and cache hits": while the target
 * verifies the current block, the drafter's packed pass drafts the successor
 * blocks; the two do not depend on each other.  d3d_async_round runs
 * d3d_packed_draft_attn (*attn) and d3d_spec_verify (*verify, with its
 * optional fused branch match) as one cooperative launch: the attention's
 * CTAs (d3d_packed_draft_attn_ctas of them) and the verification's CTAs on
 * the remaining SMs, one CTA per SM.  Outputs, workspaces, status words and
 * error codes are those of the two calls.  D3D_ERR_UNSUPPORTED when the
 * attention would split keys across CTAs or fill every SM, when a part has
 * nothing to compute, or for greedy verification (temperature 0): then make
 * the two calls on one stream: the attention (D3D_ATTN_AFTER_DEPENDENT when
 * the kernel before it may write its inputs), then the verification with an
 * sm_limit and D3D_VERIFY_AFTER_INDEPENDENT; or the verification with an
 * sm_limit, then the attention with D3D_ATTN_AFTER_INDEPENDENT.
 * Field meanings are those of the arguments of the two calls.
 * ======================================================================== */
typedef struct {
    const void *q, *k_prefix, *v_prefix, *k_packed, *v_packed;
    const d3d_segment_t *segs;
    const int32_t *cu_prefix, *cu_q, *cu_seg;
    int R, Hq, Hkv, d, max_q, max_prefix, total_q, total_prefix, total_segs;
    float scale;
    void *out;
    void *ws;
    size_t ws_bytes;
} d3d_attn_call_t;

typedef struct {
    const void *target_logits, *draft_logits;
    int logits_dtype;
    const int32_t *draft_tokens;
    const float *u_accept, *u_sample;
    int R, B, V;
    float temperature;
    int32_t *accept_len, *out_tokens, *num_tokens;
    float *alpha, *p_draft, *q_draft, *awl_weight;
    const int32_t *heads, *head_len;
    int M;
    int32_t *branch;
    void *ws;
    size_t ws_bytes;
} d3d_verify_call_t;

int d3d_async_round(const d3d_attn_call_t *attn, const d3d_verify_call_t *verify, cudaStream_t stream);

/* ========================================================================
 * Branch cache-hit match.
 *
 * [D3D] "Background: asynchronous drafting and cache hits": in the next
 * round, if the verified prefix equals the beginning of a pre-drafted
 * branch exactly, that branch's remaining draft tokens are reused.
 *
 *   branch[r] = smallest k with head_len[r,k] == verified_len[r] and
 *               heads[r,k,0:len] == verified[r,0:len]; -1 when none.
 *   verified [R, B], verified_len [R]  int32 (the verified tokens of the
 *               round, i.e. out_tokens/num_tokens of d3d_spec_verify)
 *   heads [R, M, B], head_len [R, M]   int32 (tokens past a head's length
 *               are ignored)
 *   branch [R] int32 output
 * A length outside [0, B] never matches.  No workspace.
 * ======================================================================== */
int d3d_branch_match(const int32_t *verified, const int32_t *verified_len, const int32_t *heads,
                     const int32_t *head_len, int R, int M, int B, int32_t *branch, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* D3D_H_ */
