/*
 * spec_verify.h -- C ABI of the speculative-sampling verify library for
 * NVIDIA GB300 (sm_103a).
 *
 * One vocabulary sweep per (batch row, drafted position) computes the
 * temperature softmax of target and draft logits, the overlap
 * alpha = sum_v min(p, q) = 1 - d_TV(p, q), the min(1, p/q) acceptance, the
 * residual max(0, p - q) correction and the bonus draw; the E2E-TV entry
 * point turns the same sweep into a loss and its draft-logit gradient.
 *
 * Citations name the page and the section that defines each operation:
 *   "Speculative Decoding 与 MTP：先猜多个 token，再让大模型一次验完"
 *   "读 Qwen Bebop 与 DeepSeek DSpark：Speculative Decoding 正在从技巧变成系统工程"
 *   "SpecOPD: Branch-Parallel On-Policy Distillation for Speculative Decoding"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every buffer argument is a DEVICE pointer owned by the caller.  The
 *    library allocates no device memory; scratch space is the caller's
 *    `workspace` (size from the matching *_workspace_bytes function).
 *  - Logit tensors are row-major and contiguous: element v of position k of
 *    batch row b sits at base + ((b * P + k) * V + v) * elem_size, where P is
 *    the number of positions stored per batch row.  Bulk (TMA) loads are used
 *    when V * elem_size is a multiple of 16 bytes and the base is 16-byte
 *    aligned; other shapes take a slower element-wise staging path.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  The host return value covers argument checks
 *    and the launch only.  Problems found in the data are OR-ed into the
 *    caller's 32-bit device word `dev_status` (may be NULL) and become visible
 *    once the caller synchronises the stream; kernels never trap.
 *  - The workspace must be zero-filled before its first use (for instance by
 *    cudaMemsetAsync); every call that completes leaves it zero-filled again.
 *    Two calls that may run at the same time on the GPU must not share a
 *    workspace.
 *  - Temperatures are float32; T == 0 selects greedy decoding where allowed.
 *  - Limits: B >= 0, 0 <= K <= 64, 1 <= V, and 2 * V * elem_size may not
 *    exceed 16 CTAs' worth of shared memory (V up to about 900k for bf16).
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1, /* a pointer, size, dtype or temperature is invalid */
  SPEC_ERR_UNSUPPORTED = 2, /* valid request beyond the library's limits */
  SPEC_ERR_CUDA = 3         /* the CUDA runtime reported an error */
} spec_status_t;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

/* Bits OR-ed into *dev_status by the kernels. */
#define SPEC_DEV_BAD_TOKEN 1u      /* a drafted token outside [0, V) (treated as rejected) */
#define SPEC_DEV_BAD_LOGITS 2u     /* NaN or +inf logit, or no finite logit in a row */
#define SPEC_DEV_BAD_UNIFORM 4u    /* a uniform outside [0, 1) */
#define SPEC_DEV_TIMEOUT 8u        /* a bounded wait inside a kernel gave up */
#define SPEC_DEV_EMPTY_RESIDUAL 16u /* rejection with zero residual mass: drawn from p */
#define SPEC_DEV_BAD_OFFSETS 32u   /* ragged row offsets rejected (nothing computed), or a tree parent outside [-1, i) */

/* Version of this ABI (bumped on any signature change). */
int spec_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* spec_status_string(spec_status_t status);

/* Number of kernels this library has launched in this process, over every
 * device and stream: counted on the host when a launch is enqueued without
 * error (library memsets are not counted).  For measurement: read it before
 * and after a timed region.  Never fails. */
unsigned long long spec_kernel_launches(void);

/* ------------------------------------------------------------------------ */
/* Batched verify step.
 *
 * Defined by "Speculative Decoding 与 MTP", section 2 (draft/verify loop: K
 * candidates, target distributions p_1..p_K plus the bonus distribution, the
 * first rejection ends the block), section 3 (accept with min(1, p/q); after
 * a rejection draw from the residual max(0, p - q), never from the full p)
 * and section 4 (greedy T == 0 compares with the target argmax; p and q use
 * the same temperature).  The overlap written to alpha_out is alpha_RS of
 * "读 Qwen Bebop 与 DeepSeek DSpark", section "用公式看".
 *
 * target_logits  [B, K+1, V] dtype: p_k = softmax(target[b,k] / T); row K is
 *                the bonus distribution.
 * draft_logits   [B, K, V] dtype: q_k = softmax(draft[b,k] / T).  May be NULL
 *                only when T == 0 and alpha_out == NULL.
 * draft_tokens   [B, K] int32: the drafted tokens y_k (sampled by the caller).
 * u_accept       [B, K] float32 in [0, 1): draft k is accepted iff
 *                u_accept <= p_k(y_k) / q_k(y_k).  Unused when T == 0.
 * u_final        [B] float32 in [0, 1): inverse-CDF uniform for the one
 *                correction or bonus token of the row.  Unused when T == 0.
 * out_tokens     [B, K+1] int32 (written): the n accepted drafts, then the
 *                correction (n < K) or bonus (n == K) token, then -1.
 * n_accepted     [B] int32 (written): n in [0, K]; tokens emitted = n + 1.
 * alpha_out      [B, K] float32 or NULL: per-position overlap alpha_k
 *                (at T == 0 the indicator [argmax p_k == argmax q_k]).
 * Inverse CDF: the smallest token v whose running sum in vocabulary order
 * exceeds u_final times the total mass.
 */
size_t spec_verify_workspace_bytes(int B, int K, int V);

spec_status_t spec_verify(const void* target_logits, const void* draft_logits,
                          spec_dtype_t dtype, int B, int K, int V,
                          float temperature, const int32_t* draft_tokens,
                          const float* u_accept, const float* u_final,
                          int32_t* out_tokens, int32_t* n_accepted,
                          float* alpha_out, uint32_t* dev_status,
                          void* workspace, size_t workspace_bytes,
                          void* stream);

/* ------------------------------------------------------------------------ */
/* Relaxed verify -- LOSSY: the output no longer follows the target
 * distribution.
 *
 * "Speculative Decoding 与 MTP", section 4: accepting a candidate because it
 * lies in the target's top-k, or because its logprob is close, raises the
 * acceptance rate but gives up the lossless guarantee; results must be
 * labelled lossy.  Draft k is accepted, in prefix order, when its drafted
 * token ranks among the target's top_k tokens (by logit, ties to the smaller
 * index; top_k <= 0: no rank condition) and
 * log p_k(y) >= max_v log p_k(v) - delta (delta = +inf: no gap condition).
 * The first rejected position emits a draw from the full p_k with u_final
 * (no residual); a block with every draft accepted emits the bonus from
 * p_{K+1}, as spec_verify does.  alpha_out reports the exact overlap.
 *
 * Arguments as spec_verify (same workspace size), without u_accept;
 * temperature T > 0; delta >= 0.
 */
spec_status_t spec_verify_relaxed(const void* target_logits,
                                  const void* draft_logits, spec_dtype_t dtype,
                                  int B, int K, int V, float temperature,
                                  int top_k, float delta,
                                  const int32_t* draft_tokens,
                                  const float* u_final, int32_t* out_tokens,
                                  int32_t* n_accepted, float* alpha_out,
                                  uint32_t* dev_status, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Candidate trees.
 *
 * A tree of N candidate nodes per row is given by parent[b][i] < i (-1: the
 * node hangs on the committed prefix).  "SpecOPD", section "树注意力(Tree
 * Attention)": node u may attend to v iff v is u or an ancestor of u, so one
 * batched target pass scores every node without leaking sibling branches.
 *
 * spec_tree_mask: mask [B, N, N] uint8 (written): 1 iff v is u or an
 * ancestor of u; depth [B, N] int32 or NULL: the number of strict ancestors
 * (the node's offset past the prefix).  A parent outside [-1, i) sets
 * SPEC_DEV_BAD_OFFSETS and stops that node's walk.
 */
spec_status_t spec_tree_mask(const int32_t* parent, int B, int N,
                             uint8_t* mask, int32_t* depth,
                             uint32_t* dev_status, void* stream);

/* Greedy (T = 0) verify of a candidate tree, committing one path per row:
 * "Speculative Decoding 与 MTP", section 4 (keep a candidate equal to the
 * target argmax; the first mismatch emits the target's token) and section 11
 * (a tree commits a single path).
 *
 * target_logits [B, N + 1, V] dtype: slot 0 after the committed prefix, slot
 *               i + 1 after node i (one target pass over the tree, masked as
 *               spec_tree_mask gives).
 * parent, node_tokens [B, N] int32.
 * From the prefix, the walk moves to the first child (node order) whose token
 * is the current slot's argmax (smallest index on ties), and emits that argmax
 * where no child matches.
 * path        [B, N] int32 (written): accepted nodes, prefix side first, -1 after.
 * out_tokens  [B, N + 1] int32 (written): their tokens, then the emitted
 *             target token, then -1.
 * n_accepted  [B] int32 (written): accepted nodes (-1 for a bad parent map).
 * Sampling (T > 0) over trees needs a multi-candidate acceptance rule that
 * the cited pages do not give; it is not provided.
 */
size_t spec_tree_verify_workspace_bytes(int B, int N, int V);

spec_status_t spec_tree_verify_greedy(const void* target_logits,
                                      spec_dtype_t dtype, int B, int N, int V,
                                      const int32_t* parent,
                                      const int32_t* node_tokens,
                                      int32_t* path, int32_t* out_tokens,
                                      int32_t* n_accepted,
                                      uint32_t* dev_status, void* workspace,
                                      size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Ragged verify: every row verifies its own number of drafted tokens, in
 * flattened tensors.
 *
 * "读 Qwen Bebop 与 DeepSeek DSpark", section "DSpark 真正厉害的地方：它为生产系统
 * 做了让步" (variable-length verification tokens of all requests are
 * flattened, and a marker tensor carries which request each belongs to) and
 * section "DSpark 的第二块拼图" (per-request verify lengths l_r); the
 * acceptance, correction and bonus rules are those of spec_verify.
 *
 * row_offsets  [B + 1] int32, device: row r owns flattened target rows
 *              [row_offsets[r], row_offsets[r+1]) = its l_r drafted positions
 *              then its bonus position; row_offsets[0] = 0,
 *              row_offsets[B] = units, 0 <= l_r <= 64.  Offsets that break
 *              this set SPEC_DEV_BAD_OFFSETS and nothing is computed.
 * units        the number of flattened target rows (host value).
 * target_logits [units, V] dtype; draft_logits [units - B, V] dtype, drafted
 *              row of (r, j) at row_offsets[r] - r + j (NULL if units == B).
 * draft_tokens, u_accept [units - B]: same flattened order as the drafts.
 * u_final      [B].  temperature T > 0.
 * out_tokens   [units] int32: row r's n accepted drafts, then the correction
 *              or bonus token, then -1, at row_offsets[r] ...
 * n_accepted   [B]; alpha_out [units - B] float32 or NULL.
 * The workspace follows the common rules (zero before first use, zero
 * after every call).  The per-unit marker (row, position, bonus) is built in
 * the workspace by the call.
 */
size_t spec_verify_ragged_workspace_bytes(int B, int units, int V);

spec_status_t spec_verify_ragged(const void* target_logits,
                                 const void* draft_logits, spec_dtype_t dtype,
                                 int B, const int32_t* row_offsets, int units,
                                 int V, float temperature,
                                 const int32_t* draft_tokens,
                                 const float* u_accept, const float* u_final,
                                 int32_t* out_tokens, int32_t* n_accepted,
                                 float* alpha_out, uint32_t* dev_status,
                                 void* workspace, size_t workspace_bytes,
                                 void* stream);

/* ------------------------------------------------------------------------ */
/* Allocation-free verify.  The pages have no counterpart: this entry point
 * exists for callers that cannot allocate device memory when they run a
 * verify step -- runtimes whose pool owns all device memory from start-up,
 * plugin hosts that provide buffers but no allocator, and latency-critical
 * decode loops that cannot take the device-wide synchronisation of
 * cudaMalloc / cudaFree.
 *
 * Same arguments and results as spec_verify, without the workspace: the
 * scratch is a fixed device array of SPEC_NOALLOC_SCRATCH_BYTES inside the
 * library, held by every GPU that loads the library until the process exits.
 * Sizes whose spec_verify_workspace_bytes(B, K, V) exceeds it are rejected with
 * SPEC_ERR_UNSUPPORTED (at K = 4 that is 393 rows, at K = 7 245 rows).  No call
 * allocates or frees memory; each clears the part of the array it uses with
 * cudaMemsetAsync on `stream`.
 *  - The first call on a device looks up the array's device address (once per
 *    device, with that device current; a failed lookup is retried by the next
 *    call); make that first call before any stream capture.
 *  - Every call on a device shares the one array: calls that may overlap on
 *    the GPU (different streams without ordering between them) race and give
 *    wrong results.  Serialise them. */
#define SPEC_NOALLOC_SCRATCH_BYTES (4u << 20)

spec_status_t spec_verify_noalloc(const void* target_logits,
                                  const void* draft_logits, spec_dtype_t dtype,
                                  int B, int K, int V, float temperature,
                                  const int32_t* draft_tokens,
                                  const float* u_accept, const float* u_final,
                                  int32_t* out_tokens, int32_t* n_accepted,
                                  float* alpha_out, uint32_t* dev_status,
                                  void* stream);

/* ------------------------------------------------------------------------ */
/* Overlap statistics of K drafted positions.
 *
 * alpha_k = sum_v min(p_k, q_k) = 1 - d_TV(p_k, q_k), prefix survival
 * a_j = prod_{k<=j} alpha_k and E[tau] = sum_j a_j: "读 Qwen Bebop 与
 * DeepSeek DSpark", section "用公式看" (alpha_RS, d_TV, P(tau >= j), E[tau])
 * and section "DSpark 的第二块拼图" (soft label c*_k = 1 - d_TV, a_j).
 *
 * target_logits  [B, KT, V] dtype, KT >= K: position k < K of each row is used
 *                (pass KT = K + 1 to reuse a verify batch's target tensor).
 * draft_logits   [B, K, V] dtype.
 * temperature    T >= 0 (T == 0: alpha_k = [argmax p_k == argmax q_k]).
 * alpha          [B, K] float32 (written, required).
 * tv             [B, K] float32 or NULL: 1 - alpha_k.
 * prefix_survival [B, K] float32 or NULL.
 * expected_accepted [B] float32 or NULL: E[tau] (add 1 for emitted tokens).
 */
size_t spec_overlap_workspace_bytes(int B, int K, int V);

spec_status_t spec_overlap(const void* target_logits, const void* draft_logits,
                           spec_dtype_t dtype, int B, int K, int KT, int V,
                           float temperature, float* alpha, float* tv,
                           float* prefix_survival, float* expected_accepted,
                           uint32_t* dev_status, void* workspace,
                           size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* E2E-TV loss and its gradient with respect to the draft logits.
 *
 * L = (1/B) sum_b sum_{j=1..K} prod_{k<=j} alpha_{b,k}: "读 Qwen Bebop 与
 * DeepSeek DSpark", section "Bebop 的解法" (E[tau] written with
 * 1 - d_TV(p_k, q_k)); "SpecOPD", method step (6): prefix products of the
 * per-position overlap, only the draft probabilities are differentiated and
 * the target is a constant.  The loss is the expected accepted length (to be
 * maximised); pass grad_scale = -1 to get the gradient of -L.
 *
 * grad[b,k,v] = grad_scale * dL/dalpha_{b,k} * (q_v / T) * (1[q_v < p_v] - S),
 * S = sum_{u: q_u < p_u} q_u, with
 * dL/dalpha_k = (1/B) prod_{i<k} alpha_i (1 + alpha_{k+1} + alpha_{k+1} alpha_{k+2} + ...).
 *
 * target_logits  [B, KT, V] dtype, KT >= K (first K positions used).
 * draft_logits   [B, K, V] dtype.
 * temperature    T > 0.
 * loss_out       [1] float32 (written).
 * alpha_out      [B, K] float32 or NULL.
 * grad_draft_logits [B, K, V] float32 (overwritten).
 */
size_t spec_e2e_tv_workspace_bytes(int B, int K, int V);

spec_status_t spec_e2e_tv_fwd_bwd(const void* target_logits,
                                  const void* draft_logits, spec_dtype_t dtype,
                                  int B, int K, int KT, int V,
                                  float temperature, float grad_scale,
                                  float* loss_out, float* alpha_out,
                                  float* grad_draft_logits,
                                  uint32_t* dev_status, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Per-position distribution diagnostics of K drafted positions.
 *
 * "读 Qwen Bebop 与 DeepSeek DSpark", section "Qwen Bebop：RL 里的瓶颈不是 MTP
 * 不会猜，而是策略熵在变" (acceptance falls as the target's entropy rises; a
 * point-mass drafter is accepted with probability p(argmax q)) and section
 * "Bebop 的解法" (cross-entropy or KL training of the drafter against
 * training for the acceptance itself).  With p = softmax(target / T) and
 * q = softmax(draft / T), natural logarithms, 0 log 0 = 0:
 *   alpha   = sum_v min(p_v, q_v)
 *   entropy = -sum_v p_v log p_v
 *   kl      = sum_v p_v (log p_v - log q_v)   (+inf if some q_v = 0 < p_v)
 *   cross_entropy = entropy + kl = -sum_v p_v log q_v
 *   alpha_target_only = p(y_hat), y_hat = argmax_v q_v (smallest index on ties)
 *
 * target_logits  [B, KT, V] dtype, KT >= K (first K positions used).
 * draft_logits   [B, K, V] dtype.
 * temperature    T > 0.
 * alpha, entropy, cross_entropy, kl, alpha_target_only
 *                [B, K] float32 each, or NULL (not written).
 * A row with NaN or +inf logits, or no finite logit, gets NaN in every output
 * and SPEC_DEV_BAD_LOGITS.
 */
size_t spec_diagnostics_workspace_bytes(int B, int K, int V);

spec_status_t spec_diagnostics(const void* target_logits,
                               const void* draft_logits, spec_dtype_t dtype,
                               int B, int K, int KT, int V, float temperature,
                               float* alpha, float* entropy,
                               float* cross_entropy, float* kl,
                               float* alpha_target_only, uint32_t* dev_status,
                               void* workspace, size_t workspace_bytes,
                               void* stream);

/* ------------------------------------------------------------------------ */
/* Top-k / top-p truncation of logit rows, to be applied with the same
 * arguments to the target and the draft logits before a verify step.
 *
 * "Speculative Decoding 与 MTP", section 4 (p and q are both computed after the
 * agreed temperature and top-k / top-p transforms) and section 23 (a mask that
 * only one side applies breaks correctness).  Tokens are ranked by logit,
 * larger first, ties to the smaller index.  Top-k (0 < top_k < V) keeps the
 * first top_k.  Top-p (top_p < 1) then renormalises softmax(z / T) over the
 * kept tokens and keeps the shortest ranked prefix whose mass reaches top_p.
 * Dropped logits become -inf; kept logits are copied unchanged.
 *
 * logits       [rows, V] dtype, device.
 * out          [rows, V] dtype, device; may be `logits` itself (in place) but
 *              may not overlap it otherwise.
 * temperature  T > 0 when top_p < 1 (unused otherwise).
 * top_k        >= 0; 0 or >= V disables top-k.
 * top_p        in (0, 1]; 1 disables top-p.
 * A row holding a NaN or +inf logit, or no finite logit, is copied unchanged
 * and sets SPEC_DEV_BAD_LOGITS.  Top-p masses are fixed point with 2^-44 of
 * the row maximum's mass as unit; a cut whose preceding mass lies within
 * about 1e-6 of top_p may move by one token against exact arithmetic.
 */
spec_status_t spec_truncate_logits(const void* logits, void* out,
                                   spec_dtype_t dtype, int rows, int V,
                                   float temperature, int top_k, float top_p,
                                   uint32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Verify-length scheduling.
 *
 * "读 Qwen Bebop 与 DeepSeek DSpark", section "DSpark 的第二块拼图：置信度调度验证
 * 长度": request r verifying l_r drafted tokens adds 1 + l_r tokens to the
 * target batch, B = sum_r (1 + l_r), and produces tau_r = 1 +
 * sum_{j<=l_r} a_{r,j} tokens in expectation; the lengths maximise
 * Theta = (sum_r tau_r) * SPS(B), SPS(B) the engine's decode steps per second
 * at batch B.  For a fixed B the best choice takes the B - R largest
 * survivals; equal survivals are taken in (row, position) order and equal
 * Theta keeps the smaller B.
 *
 * survival   [R, L] float32: a_{r,j}, j = 1..L, non-increasing in j (the
 *            prefix_survival output of spec_overlap is such a table); the
 *            running minimum along j is used; NaN counts as 0 and sets
 *            SPEC_DEV_BAD_LOGITS.
 * sps        [sps_len] float32 >= 0: SPS(B) for B = 0 .. sps_len - 1,
 *            sps_len >= R * (1 + L) + 1.
 * lengths    [R] int32 (written): l_r in [0, L].
 * objective  [2] float32 or NULL: {Theta, tau} at the choice.
 * Limits: 1 <= L <= 64 and R * L <= 16384 (SPEC_ERR_UNSUPPORTED beyond).
 * One cluster of 16 CTAs (distributed shared memory; no workspace).
 * Survivals are summed exactly as integers in units of 2^-48 (one
 * rounding each, so sums of n of them are within n * 2^-49 of the real sum);
 * Theta is formed in fp64.  A choice whose Theta lies within about 1e-10
 * relative of another B's may therefore differ from exact arithmetic.
 */
spec_status_t spec_schedule_lengths(const float* survival, int R, int L,
                                    const float* sps, int sps_len,
                                    int32_t* lengths, float* objective,
                                    uint32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Failure-path self-test of the bounded wait.
 *
 * Launches one warp that waits, with the same bounded mbarrier wait the
 * sweep uses on its bulk copies, for a phase of a fresh shared-memory
 * mbarrier that nothing ever completes.  No copy is in flight.  After
 * limit_ns nanoseconds of wall time the wait gives up, and the kernel ORs
 * SPEC_DEV_TIMEOUT into *dev_status and returns.  Tests use it to check that
 * a wait that runs out is reported on the status word and that the context
 * stays usable afterwards.
 * limit_ns   in [1, 10^10] (10 s).
 * dev_status [1] uint32, device (required).
 * Returns SPEC_ERR_INVALID_ARG for a limit out of range or a NULL status.
 */
spec_status_t spec_selftest_bounded_wait(uint64_t limit_ns, uint32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Launch shape the library picks for a sampling verify sweep over `units`
 * (row, position) pairs of V logits with rows on 16-byte boundaries (for
 * benchmarks and diagnostics; the two-pass sweep when units x 2 rows reach
 * 200 MB, as in spec_set_kernel_override): CTAs per cluster, threads per CTA (608 for
 * the two-pass sweep: sixteen consumer warps, a copy warp, a decision warp
 * and a completion warp; 256 for the single-read sweep), dynamic shared memory
 * per CTA, the number of persistent clusters launched and the shared-memory
 * stages per CTA.  Needs a current CUDA device.  Returns
 * SPEC_ERR_UNSUPPORTED if V does not fit.  Any output pointer may be NULL. */
spec_status_t spec_launch_shape(spec_dtype_t dtype, int units, int V,
                                int* cluster_ctas, int* threads,
                                int* smem_bytes, int* clusters, int* stages);

/* Forces the CTAs per cluster (1..16) and caps the shared-memory stages per
 * CTA (the two-pass sweep's ring stages, at least 1; the single-read sweep's
 * 1 or 2) of later launches in this process, for launch-shape sweeps in
 * benchmarks; 0 restores the automatic choice of either.  Process-wide; not
 * synchronised with launches in flight. */
void spec_set_launch_override(int cluster_ctas, int stages);

/* Selects the vocabulary-sweep kernel of later verify, overlap and E2E-TV
 * calls in this process: 0 automatic (the two-pass sweep for calls that read
 * at least 200 MB of logits, where rows start on 16-byte boundaries and the
 * mode has it; else the single-read sweep),
 * 1 the single-read sweep (rows resident in cluster shared memory between
 * passes), 2 the two-pass sweep where it applies (pass A from HBM, pass C
 * from L2).  Any other value means 0.  For tests and benchmarks; both give
 * the same results within the parity bar.  Process-wide; not synchronised
 * with launches in flight. */
void spec_set_kernel_override(int kernel);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
