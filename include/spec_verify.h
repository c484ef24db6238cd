/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) batched speculative-sampling
 * verifier.
 *
 * The operation (sources cited by page title and section):
 *   - "深入推测解码：从概念到实现" (Exploring Speculative Decoding), section
 *     保证原始分布: accept a drafted token x with probability
 *     min(1, p(x)/q(x)); on rejection resample from max(0, p(x) - q(x)).
 *   - "RTP-LLM Speculative Engine 深度解析", section 拒绝采样算法: test the
 *     drafts in order, stop at the first rejection.
 *   - "投机采样" (razer666.cn), sections 第三步 to 第五步 of 投机解码算法 and
 *     the output-length cases: the correction is drawn from
 *     norm(max(0, p_{n+1} - q_{n+1})); when all gamma drafts are accepted one
 *     more token is drawn from p_{gamma+1}, so 1..gamma+1 tokens come out;
 *     section 验收标准 / 精确匹配: the greedy variant accepts a draft iff it is
 *     the target's most probable token.
 *
 * Conventions shared by every entry point:
 *   - All tensor arguments are DEVICE pointers to dense row-major arrays,
 *     owned by the caller.  The library allocates nothing, keeps no state
 *     between calls and never synchronises: every call only enqueues work on
 *     `stream` and returns.
 *   - Shapes: B requests, K draft positions per request (0 <= K <= 31),
 *     vocabulary V (8 <= V <= 2^24, V a multiple of 8).
 *   - Host-checkable errors are returned before anything is enqueued.
 *   - Data errors are found on the device (see SPEC_BADBIT_*): the offending
 *     request gets out_ids[b, :] = -1 and out_num_accepted[b] = -1, a bit is
 *     OR-ed into the device status word, and other requests are unaffected.
 *     No kernel traps.
 *   - Calls that share a workspace must not overlap on the GPU (issue them on
 *     one stream, or order the streams).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st* spec_stream_t;
typedef struct CUevent_st* spec_event_t;  /* a cudaEvent_t */

typedef enum {
    SPEC_OK = 0,
    SPEC_ERR_INVALID_ARG = 1, /* null pointer, negative size, K > 31, ... */
    SPEC_ERR_UNSUPPORTED = 2, /* V not a multiple of 8, V out of range, misaligned pointer */
    SPEC_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    SPEC_ERR_WORKSPACE = 4    /* workspace too small or not 256-byte aligned */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

#define SPEC_MAX_K 31

/* Bits of the device status word (0 when every request was well formed). */
#define SPEC_BADBIT_NUM_DRAFT 1u   /* num_draft[b] outside [0, K] */
#define SPEC_BADBIT_TEMPERATURE 2u /* temperature[b] NaN, negative or infinite */
#define SPEC_BADBIT_DRAFT_ID 4u    /* draft_ids[b, j] outside [0, V) for some j < num_draft[b] */
#define SPEC_BADBIT_EMPTY_ROW 8u   /* a sampling row j <= num_draft[b] whose logits are all -inf */
#define SPEC_BADBIT_NO_PROBS 16u   /* a sampling request with drafts but draft_probs == NULL */
#define SPEC_BADBIT_TIMEOUT 32u    /* an internal bounded wait gave up (never expected) */
#define SPEC_BADBIT_TREE 64u       /* spec_verify_tree: a node whose parent is not an earlier node */

/* Human-readable name of a status code (static string). */
const char* spec_status_str(spec_status s);

/* Bytes of scratch memory spec_verify needs for these sizes (0 on bad sizes).
 * The workspace must be 256-byte aligned; its contents need no
 * initialisation and are overwritten by every call. */
size_t spec_verify_workspace_size(int B, int K, int V);

/*
 * spec_verify -- verify K drafted tokens for each of B requests.
 *
 *   target_logits    [B, K+1, V], dtype logits_dtype (f32 or bf16), 16-byte
 *                    aligned.  Row (b, j) is the target model's logits for the
 *                    position that drafted token j would fill; row K (or row
 *                    num_draft[b]) is the bonus position.  Rows j > num_draft[b]
 *                    are never read.  Each logit is finite or -inf (a
 *                    masked token); +inf and NaN logits are outside the
 *                    contract (the row's outputs are then unspecified, and
 *                    no kernel indexes memory by a logit value).
 *   draft_probs      [B, K, V] float32, 16-byte aligned: the draft
 *                    distribution q_j that drew draft token j, used as given
 *                    (not renormalised).  Only row e_b (the first rejected
 *                    position) is read whole; elsewhere only q_j(x_j).  May be
 *                    NULL when no sampling request has a draft.
 *   draft_ids        [B, K] int32: x_j; entries j >= num_draft[b] are ignored.
 *   num_draft        [B] int32: n_b in [0, K] drafts to verify for request b.
 *   temperature      [B] float32: T_b = 0 selects greedy exact-match
 *                    verification; T_b > 0 samples from p = softmax(l / T_b).
 *   seed             Philox4x32-10 key (low word, high word).  Row j of
 *                    request b draws the block at counter (b, j, 0, 0): lane 0
 *                    is the acceptance uniform, lane 1 the uniform of a token
 *                    emitted from that row, each mapped to ((x >> 8) + 1) 2^-24.
 *                    Change the seed between calls.
 *   out_ids          [B, K+1] int32 (written): the a_b accepted drafts, then the
 *                    emitted token (resampled correction, bonus token, or the
 *                    greedy target token), then -1.
 *   out_num_accepted [B] int32 (written): a_b in [0, n_b], or -1 for a bad
 *                    request.
 *   workspace        scratch of at least spec_verify_workspace_size(B, K, V)
 *                    bytes, 256-byte aligned; the device status word lives in
 *                    it (spec_verify_status_ptr).
 *   stream           stream the kernels are enqueued on.
 *
 * The call runs one of two verifiers with the same arithmetic and the same
 * uniforms, whichever is faster for the batch (spec_verify_path tells which):
 *   - request by request (spec_verify_by_request), once B is at least 2.1
 *     times the device's SM count: request b is verified the way the pages'
 *     loop runs ("RTP-LLM Speculative Engine", 拒绝采样算法: test draft j,
 *     break at the first rejection), so rows 0..a_b are read, rows after the
 *     first rejection never are, and the rejected row is read a second time
 *     for the residual.  Two kernels: a one-CTA set-up kernel, then one
 *     persistent CTA per SM.
 *   - every row 0..n_b in one pass spread over the whole GPU
 *     (spec_verify_all_rows), for smaller batches, and whenever V exceeds
 *     96 * 2048 tokens or no CTA of the request-by-request kernel fits an SM.
 *     Five kernels.
 * Both give identical out_ids and out_num_accepted on valid inputs.  Every
 * draft id j < n_b is range-checked first; a sampling row that the verifier
 * reads and that holds no finite logit makes the request bad
 * (SPEC_BADBIT_EMPTY_ROW): request by request checks rows 0..a_b, the
 * all-rows pass rows 0..n_b.  The call never synchronises.
 *
 * Sampling: p_j = softmax(l_j / T_b) is computed in float32 with float64
 * accumulation; accept x_j iff p_j(x_j) > 0 and (q_j(x_j) == 0 or
 * u_j <= p_j(x_j) / q_j(x_j)); a_b = the number of leading accepted drafts;
 * if a_b < n_b the token at a_b is the smallest x with
 * sum_{y<=x} max(0, p(y) - q(y)) >= u' * sum_y max(0, p(y) - q(y)) on row a_b
 * (falling back to p if that residual has no mass); if a_b = n_b it is drawn
 * the same way from p_{n_b}.  Greedy: x_j is accepted iff it is the lowest
 * index of the maximum of l_j; the emitted token is that argmax of row a_b.
 */
spec_status spec_verify(const void* target_logits, spec_dtype logits_dtype,
                        const float* draft_probs, const int32_t* draft_ids,
                        const int32_t* num_draft, const float* temperature, uint64_t seed,
                        int B, int K, int V, int32_t* out_ids, int32_t* out_num_accepted,
                        void* workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_verify_ex -- spec_verify plus sharding and diagnostics.
 *   request_offset  added to b in the Philox counter, so that a shard holding
 *                   requests [o, o + B) of a larger batch draws the same
 *                   uniforms as the unsharded call.
 *   dbg_rows        [B, K+1, 4] float32 or NULL: per row j < n_b of a sampling
 *                   request {p_j(x_j), u_j, Z_j, accepted (1/0)}, where Z_j =
 *                   sum_x exp((l_j(x) - max l_j) / T_b); greedy rows give
 *                   {NaN, NaN, NaN, accepted}; untested rows {NaN, NaN, NaN, -1}.
 *   dbg_req         [B, 4] float32 or NULL: {mode, emission row, emission mass,
 *                   u'}; mode -1 bad, 0 greedy, 1 residual, 2 bonus,
 *                   3 residual without mass (drawn from p), 4 typical
 *                   acceptance (drawn from p, spec_verify_typical only).
 *   dev_status      int32 device word or NULL: receives the status bits of
 *                   this call (zeroed by the call itself).
 */
spec_status spec_verify_ex(const void* target_logits, spec_dtype logits_dtype,
                           const float* draft_probs, const int32_t* draft_ids,
                           const int32_t* num_draft, const float* temperature, uint64_t seed,
                           int B, int K, int V, int32_t* out_ids, int32_t* out_num_accepted,
                           void* workspace, size_t workspace_bytes, spec_stream_t stream,
                           uint32_t request_offset, float* dbg_rows, float* dbg_req,
                           int32_t* dev_status);

/*
 * spec_verify_typical -- the lossy typical-acceptance rule ("投机采样",
 * section 验收标准, item Typical Acceptance: a draft token is kept when the
 * target's probability of it reaches a hard threshold, and the longest run of
 * kept drafts is taken).
 *
 * Same arguments, layout, workspace and errors as spec_verify_ex, without
 * draft_probs (the rule reads no draft distribution) and with
 *   threshold  the hard threshold theta; NaN is SPEC_ERR_INVALID_ARG, any
 *              other value (including +-inf) is allowed.
 * Sampling request b: p_j = softmax(l_j / T_b) in float32 with float64
 * accumulation; x_j is kept iff p_j(x_j) > 0 and p_j(x_j) >= theta;
 * a_b = the number of leading kept drafts; the token at position a_b (after
 * a refused draft, or the bonus token when all n_b are kept) is the smallest x
 * with sum_{y<=x} p_{a_b}(y) >= u' on row a_b, u' = lane 1 of the Philox
 * block of row a_b.  Greedy requests (T_b = 0) are verified by exact match
 * exactly as in spec_verify.  dbg_rows give {p_j(x_j), NaN, Z_j, kept};
 * dbg_req mode 4 for every sampling request.
 */
spec_status spec_verify_typical(const void* target_logits, spec_dtype logits_dtype,
                                const int32_t* draft_ids, const int32_t* num_draft,
                                const float* temperature, float threshold, uint64_t seed,
                                int B, int K, int V, int32_t* out_ids,
                                int32_t* out_num_accepted, void* workspace,
                                size_t workspace_bytes, spec_stream_t stream,
                                uint32_t request_offset, float* dbg_rows, float* dbg_req,
                                int32_t* dev_status);

/*
 * spec_verify_dev_seed -- spec_verify_ex with the Philox seed read from
 * device memory (*seed_dev, 8-byte aligned) when the kernels run instead of
 * passed by value.  A call enqueues a fixed sequence of kernels, allocates
 * nothing and never synchronises, so it can be captured once in a CUDA graph
 * and replayed for every decoding step, the caller writing the step's seed to
 * *seed_dev before each replay; replaying saves the launch gaps between the
 * kernels.  The pages have no counterpart to this entry point.  A NULL or
 * misaligned seed_dev is SPEC_ERR_INVALID_ARG; otherwise as spec_verify_ex.
 */
spec_status spec_verify_dev_seed(const void* target_logits, spec_dtype logits_dtype,
                                 const float* draft_probs, const int32_t* draft_ids,
                                 const int32_t* num_draft, const float* temperature,
                                 const uint64_t* seed_dev, int B, int K, int V, int32_t* out_ids,
                                 int32_t* out_num_accepted, void* workspace,
                                 size_t workspace_bytes, spec_stream_t stream,
                                 uint32_t request_offset, float* dbg_rows, float* dbg_req,
                                 int32_t* dev_status);

/*
 * spec_verify_early_exit -- spec_verify_ex that stops reading a request's rows
 * at its first rejection ("RTP-LLM Speculative Engine", 拒绝采样算法: the
 * per-draft loop breaks at the first rejected token, so no later position of
 * that request is ever scored).
 *
 * The call runs K + 1 passes over the logits: pass r reads row r of exactly
 * the requests that kept drafts 0..r-1 (all requests in pass 0), tests draft r
 * (or, at r = num_draft[b], takes the bonus row) and drops every request that
 * ends there.  The rows a request does read get the same arithmetic and the
 * same Philox uniforms as in spec_verify, so every output equals spec_verify's
 * on the same inputs, with two differences in what is checked: every draft id
 * is range-checked before the first pass (as spec_verify does), but a
 * sampling row that is never read is never checked for being all -inf (in
 * spec_verify such a row anywhere in 0..num_draft[b] makes the request bad),
 * and dbg_rows entries of rows that were not read hold NaN with accept = -1.
 * Logit bytes read: sum over requests of (a_b + 1) * V * elem_size, against
 * (num_draft[b] + 1) * V * elem_size for spec_verify; the price is K + 1
 * dependent kernel launches instead of one.  seed_dev: NULL (the seed is
 * `seed`), or an 8-byte aligned device pointer read in its place when the
 * kernels run, as in spec_verify_dev_seed (for CUDA graph replay; misaligned
 * is SPEC_ERR_INVALID_ARG).  Other arguments, workspace
 * (spec_verify_workspace_size), errors and the device status word as
 * spec_verify_ex.
 */
spec_status spec_verify_early_exit(const void* target_logits, spec_dtype logits_dtype,
                                   const float* draft_probs, const int32_t* draft_ids,
                                   const int32_t* num_draft, const float* temperature,
                                   uint64_t seed, int B, int K, int V, int32_t* out_ids,
                                   int32_t* out_num_accepted, void* workspace,
                                   size_t workspace_bytes, spec_stream_t stream,
                                   uint32_t request_offset, float* dbg_rows, float* dbg_req,
                                   int32_t* dev_status, const uint64_t* seed_dev);

/*
 * spec_verify_all_rows -- the verification of spec_verify_ex, every row
 * 0..num_draft[b] of every request read in one streaming pass.
 *
 * The pages' loop stops at the first rejection; this verifier reads the rows
 * after it as well, so that the whole batch's row statistics come from one
 * pass over the logits spread evenly over the GPU, then runs the acceptance
 * tests, the residual masses and the draws as four more kernels.  Its outputs
 * equal spec_verify's on the same inputs, except that every sampling row
 * 0..num_draft[b] is checked for a finite logit (a row without one makes the
 * request bad even if it lies after the first rejection), and dbg_rows hold
 * {p_j(x_j), u_j, Z_j, accepted} for every draft row j < n_b of a sampling
 * request.  Logit bytes read: sum_b (n_b + 1) V elem_size.
 *   seed_dev  NULL (the seed is `seed`) or an 8-byte aligned device pointer
 *             read in its place when the kernels run (for CUDA graph replay).
 *   events    NULL, or six CUDA events recorded as in spec_verify_profiled.
 * Other arguments, workspace (spec_verify_workspace_size), errors and the
 * device status word as spec_verify_ex.
 */
spec_status spec_verify_all_rows(const void* target_logits, spec_dtype logits_dtype,
                                 const float* draft_probs, const int32_t* draft_ids,
                                 const int32_t* num_draft, const float* temperature,
                                 uint64_t seed, int B, int K, int V, int32_t* out_ids,
                                 int32_t* out_num_accepted, void* workspace,
                                 size_t workspace_bytes, spec_stream_t stream,
                                 uint32_t request_offset, float* dbg_rows, float* dbg_req,
                                 int32_t* dev_status, const uint64_t* seed_dev,
                                 spec_event_t* events);

/*
 * spec_verify_by_request -- the verification of spec_verify_ex request by
 * request at any B ("RTP-LLM Speculative Engine", 拒绝采样算法: each request's
 * drafts tested in order, stopping at the first rejection): one persistent
 * CTA per SM claims whole requests, most drafts first, and reads a request's
 * rows 0..a_b, then the rejected row again for the residual.  Logit bytes
 * read: sum_b (a_b + 1) V elem_size, plus V * 4 for the q row of each
 * residual draw.  dbg_rows hold NaN and accept = -1 for the rows after a_b,
 * which are never read.  Falls back to the all-rows pass where its kernel
 * does not apply (V > 96 * 2048, or no CTA fits an SM).  Arguments, events,
 * workspace, errors and the device status word as spec_verify_all_rows.
 */
spec_status spec_verify_by_request(const void* target_logits, spec_dtype logits_dtype,
                                   const float* draft_probs, const int32_t* draft_ids,
                                   const int32_t* num_draft, const float* temperature,
                                   uint64_t seed, int B, int K, int V, int32_t* out_ids,
                                   int32_t* out_num_accepted, void* workspace,
                                   size_t workspace_bytes, spec_stream_t stream,
                                   uint32_t request_offset, float* dbg_rows, float* dbg_req,
                                   int32_t* dev_status, const uint64_t* seed_dev,
                                   spec_event_t* events);

/*
 * spec_verify_path -- which verifier spec_verify (and spec_verify_ex,
 * _profiled, _dev_seed, _noalloc) runs for these sizes on the current device:
 * 1 request by request, 0 the all-rows pass, -1 invalid sizes or dtype, or a
 * CUDA error while reading the device's properties.
 */
int spec_verify_path(int B, int K, int V, spec_dtype logits_dtype);

/*
 * spec_lmhead_logits -- the target's logits from its last hidden states: the
 * vocabulary projection of the one target pass that scores the drafts
 * ("投机采样", 第二步: one forward of the target yields p_1 .. p_{gamma+1};
 * "深入推测解码" 保证原始分布 step 2), on the tcgen05 tensor cores.
 *
 *   hidden      [rows, H] bf16, row-major, 16-byte aligned (device).
 *   lm_head     [V, H] bf16, row-major (token v's output embedding), aligned.
 *   logits_out  [rows, V] bf16 (written): logits[r, v] = sum_h hidden[r, h] *
 *               lm_head[v, h], products and sums in float32, rounded once to
 *               bf16 (nearest, ties to even).
 *   dev_status  one device int32; SPEC_BADBIT_TIMEOUT is or-ed in if a wait
 *               of the kernel ran out (the outputs are then incomplete).
 * H must be a multiple of 64 and V of 8 (else SPEC_ERR_UNSUPPORTED);
 * 1 <= H <= 65536, V <= 2^24, rows <= 2^24.  Enqueues one kernel on
 * `stream`; allocates nothing and does not synchronise.
 */
spec_status spec_lmhead_logits(const void* hidden, const void* lm_head, int rows, int H, int V,
                               void* logits_out, int32_t* dev_status, spec_stream_t stream);

/*
 * spec_verify_lmhead -- spec_verify_ex with the target logits produced inside
 * the call from the target's last hidden states (the fused logits producer):
 * the rows the verifier reads (j <= num_draft[b]) are projected by the
 * tcgen05 LM-head GEMM of spec_lmhead_logits, and the same kernel's epilogue
 * takes, from the bf16 logits it stores, the row statistics and the
 * acceptance that spec_verify's row pass would take.  The logits make one
 * trip to HBM (written) instead of two (written by a separate GEMM, then
 * read back).
 *
 *   hidden      [B, K+1, H] bf16 (row j of request b: the hidden state whose
 *               projection is target_logits[b, j] of spec_verify).
 *   lm_head     [V, H] bf16.
 *   logits_out  [B, K+1, V] bf16 (written for the rows read, left as it was
 *               elsewhere); the residual and bonus draws read it afterwards.
 *   workspace   at least spec_verify_lmhead_workspace_size(B, K, V, H) bytes.
 * Other arguments, outputs and errors as spec_verify_ex with bf16 logits;
 * H must be a multiple of 64 (else SPEC_ERR_UNSUPPORTED).  The outputs equal
 * spec_verify's on logits_out up to the float32 summation order of the row
 * statistics.
 */
size_t spec_verify_lmhead_workspace_size(int B, int K, int V, int H);
spec_status spec_verify_lmhead(const void* hidden, const void* lm_head, int H, void* logits_out,
                               const float* draft_probs, const int32_t* draft_ids,
                               const int32_t* num_draft, const float* temperature, uint64_t seed,
                               int B, int K, int V, int32_t* out_ids, int32_t* out_num_accepted,
                               void* workspace, size_t workspace_bytes, spec_stream_t stream,
                               uint32_t request_offset, float* dbg_rows, float* dbg_req,
                               int32_t* dev_status);

/*
 * spec_verify_tree -- token-tree verification ("投机采样", section 验证方案:
 * candidate draft sequences that share a prefix are merged into a trie, and
 * the target scores every node in one pass; SpecInfer's token-tree verifier).
 *
 * Per request b the trie has n_b = num_nodes[b] nodes, 1 <= n_b <= N <= 32;
 * node 0 is the accepted context (the root), node c >= 1 carries the draft
 * token tree_tokens[b, c] and the parent tree_parents[b, c], an earlier node
 * (0 <= parent < c).  Entries of node 0 and of nodes >= n_b are ignored.
 *   target_logits [B, N, V] f32 | bf16, 16-byte aligned: row v = the target's
 *                 logits of the token that follows node v's prefix.
 *   draft_probs   [B, N, V] f32 or NULL: row c = the draft distribution node
 *                 c's token was drawn from (row 0 unused).  NULL is allowed
 *                 when no sampling request has a child.
 *   tree_tokens, tree_parents [B, N] int32; num_nodes [B] int32;
 *   temperature   [B] f32: 0 = greedy, > 0 sampling.
 *   out_ids       [B, N] int32 (written): the tokens of the accepted path
 *                 (root excluded), then the emitted token, then -1.
 *   out_num_accepted [B] (written): the path length a_b, or -1 (bad request).
 *   out_last_node [B] (written): the last accepted node (0: none), or -1.
 * Greedy (T = 0, exact match): from v = 0, the first child of v (in node
 * index order) whose token is the lowest-index argmax of row v is accepted;
 * else that argmax is emitted.  Sampling: the children of v are tested in
 * index order against a running target r, r = p_v = softmax(l_v / T) first:
 * child c is kept iff r(x_c) > 0 and (q_c(x_c) == 0 or u_c <= r(x_c) /
 * q_c(x_c)); after a rejection r becomes max(0, r - q_c) normalised (kept as
 * it was if that has no mass).  When no child is kept the emitted token is the
 * smallest x whose prefix sum of the last residual (of r if it had no mass,
 * of p_v at a node without children) reaches u' times its total.  u_c is lane
 * 0 of the Philox block of row c - 1 and u' lane 1 of the block of row v
 * (rows as in spec_verify, request index b + request_offset), so a trie with
 * one child per node gives exactly the result of spec_verify on the chain.
 * Workspace: spec_verify_tree_workspace_size(B, N, V) bytes, 256-byte
 * aligned.  Errors as spec_verify_ex; a node whose parent is not an earlier
 * node sets SPEC_BADBIT_TREE, a token outside [0, V) SPEC_BADBIT_DRAFT_ID,
 * num_nodes outside [1, N] SPEC_BADBIT_NUM_DRAFT.  dbg_nodes [B, N, 4] (per
 * tested child c: {r(x_c), u_c, q_c(x_c), kept}; greedy: {NaN, NaN, NaN,
 * kept}) and dbg_req [B, 4] ({mode, last node, emission mass, u'}) may be
 * NULL.  N > 32 is SPEC_ERR_UNSUPPORTED.
 */
size_t spec_verify_tree_workspace_size(int B, int N, int V);
spec_status spec_verify_tree(const void* target_logits, spec_dtype logits_dtype,
                             const float* draft_probs, const int32_t* tree_tokens,
                             const int32_t* tree_parents, const int32_t* num_nodes,
                             const float* temperature, uint64_t seed, int B, int N, int V,
                             int32_t* out_ids, int32_t* out_num_accepted,
                             int32_t* out_last_node, void* workspace, size_t workspace_bytes,
                             spec_stream_t stream, uint32_t request_offset, float* dbg_nodes,
                             float* dbg_req, int32_t* dev_status);

/*
 * spec_verify_profiled -- spec_verify with timing marks: the caller's CUDA
 * events events[0..5] (cudaEvent_t) are recorded on `stream` around the
 * kernels of the call, so that events[i] -> events[i+1] brackets kernel i.
 * The request-by-request verifier runs two kernels: events[0] -> events[1]
 * brackets the set-up kernel, events[1] -> events[2] the verifier, and
 * events[2..5] are recorded together after it.  The all-rows verifier (see
 * spec_verify_all_rows, which takes the same events) runs five: plan; row
 * statistics; acceptance tests; residual masses; sampled tokens.
 * The marks separate the kernels, which otherwise overlap their launch with
 * the previous kernel's tail.  Returns SPEC_ERR_INVALID_ARG if any event is
 * NULL; otherwise as spec_verify.
 */
spec_status spec_verify_profiled(const void* target_logits, spec_dtype logits_dtype,
                                 const float* draft_probs, const int32_t* draft_ids,
                                 const int32_t* num_draft, const float* temperature,
                                 uint64_t seed, int B, int K, int V, int32_t* out_ids,
                                 int32_t* out_num_accepted, void* workspace,
                                 size_t workspace_bytes, spec_stream_t stream,
                                 spec_event_t* events);

/*
 * spec_verify_noalloc -- spec_verify without a caller-provided workspace, for
 * callers that must not allocate device memory at all: for example code
 * running inside an engine that has already handed every byte of the GPU to
 * its own pools (weights, KV cache) and forbids further cudaMalloc, or a
 * plugin whose host passes it only its input and output buffers.  For them a
 * cudaMalloc either fails or stalls the device in the middle of a decoding
 * step.  (The source pages describe no such entry point; it is an addition of
 * this library.)
 *
 * Arguments and results are those of spec_verify.  The scratch memory is one
 * array of SPEC_NOALLOC_SCRATCH_BYTES bytes of static device memory inside the
 * library, present on every GPU that loads the library until the process
 * exits; this call allocates nothing.  Sizes whose workspace
 * (spec_verify_workspace_size) exceeds SPEC_NOALLOC_SCRATCH_BYTES are rejected
 * with SPEC_ERR_WORKSPACE before anything is enqueued.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls on a device share the one array: calls that overlap on
 * the GPU (different streams, not ordered) race on it and give undefined
 * results.  The array keeps the previous call's contents, which the kernels
 * never rely on (every call rewrites what it reads).
 */
#define SPEC_NOALLOC_SCRATCH_BYTES (8u << 20)
spec_status spec_verify_noalloc(const void* target_logits, spec_dtype logits_dtype,
                                const float* draft_probs, const int32_t* draft_ids,
                                const int32_t* num_draft, const float* temperature, uint64_t seed,
                                int B, int K, int V, int32_t* out_ids, int32_t* out_num_accepted,
                                spec_stream_t stream);

/* Device address of the status word inside a workspace (no GPU work). */
int32_t* spec_verify_status_ptr(void* workspace);

/*
 * spec_verify_host -- spec_verify for callers whose inputs and outputs live in
 * host memory.  The inputs are copied to the caller's device buffers
 * (d_logits [B, K+1, V], d_probs [B, K, V], d_small: at least
 * spec_verify_host_small_bytes(B, K) bytes, 256-byte aligned), the verifier
 * runs, and out_ids / out_num_accepted are copied back, all enqueued on
 * `stream`.  When h_logits (and h_probs) are page-locked and mapped into the
 * device's address space (cudaHostAlloc / cudaHostRegister memory on a
 * unified-addressing system), copy kernels move only what the verifier
 * reads: the logits rows 0..num_draft[b], q_j(x_j) for every draft, and,
 * once the acceptances are known, the q row of each residual draw; the rest
 * of d_logits / d_probs is left as it was.  Other host memory is copied
 * whole (one cudaMemcpyAsync per tensor; pageable memory makes those copies
 * synchronous).  The call does not synchronise, so the host outputs are
 * valid after the stream is synchronised.  h_probs / d_probs may be NULL
 * when every request is greedy.
 */
size_t spec_verify_host_small_bytes(int B, int K);
spec_status spec_verify_host(const void* h_logits, spec_dtype logits_dtype, const float* h_probs,
                             const int32_t* h_draft_ids, const int32_t* h_num_draft,
                             const float* h_temperature, uint64_t seed, int B, int K, int V,
                             int32_t* h_out_ids, int32_t* h_out_num_accepted, void* d_logits,
                             float* d_probs, void* d_small, void* workspace,
                             size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_philox_fill -- the library's Philox4x32-10 for cross-checking:
 * out[4i..4i+3] = Philox4x32-10(counter = ctrs[4i..4i+3], key = (seed lo,
 * seed hi)) for i < n.  ctrs and out are device arrays of 4n uint32.
 * Source: J. Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3",
 * SC'11 (Philox4x32 with 10 rounds).
 */
spec_status spec_philox_fill(uint64_t seed, const uint32_t* ctrs, int64_t n, uint32_t* out,
                             spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
