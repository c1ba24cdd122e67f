/*
 * tva.h - tree-verification attention and greedy tree acceptance (C ABI).
 *
 * The operation (LongSpec, "Fast Tree Attention" section, Hybrid Tree Attention):
 * every query of a speculative draft tree attends (1) without a mask to the cached
 * prefix pairs {K_cache, V_cache} and (2) to the tree's own pairs {K_specs, V_specs}
 * under the tree mask, which lets a node see only its ancestors ("Faster decoding",
 * section "Chains and trees consume work differently").  The partial results are
 * combined exactly through their log-sum-exp (same LongSpec section, "Aggregation",
 * and its appendix "Correctness of attention aggregation").  The greedy verification
 * contract ("Faster decoding", section on modified rejection sampling, paragraph on
 * greedy verification) keeps the longest draft path that agrees with the target's
 * greedy tokens and emits the target's token after it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers are DEVICE pointers unless a comment says otherwise.  The caller owns
 *   every buffer; the library never allocates on these paths, except the one
 *   convenience form that says so (tree_verify_attn), whose workspace tva_release()
 *   frees.
 * - All tensors are dense, row-major and contiguous; floating-point base pointers
 *   must be 16-byte aligned.  Shapes use: B batch, Hq query heads, Hkv KV heads
 *   (Hq % Hkv == 0, query head h reads KV head h / (Hq / Hkv)), d head_dim,
 *   P_b prefix length of sequence b, m_b tree size of sequence b, N = sum of m_b.
 * - Trees: parent[] holds LOCAL node ids; parent[i] == -1 makes node i a child of
 *   the prefix end; otherwise 0 <= parent[i] < i (topological order).  A node sees
 *   its ancestors and itself.
 * - Work is enqueued asynchronously on `stream` (a cudaStream_t; 0 = legacy default
 *   stream).  Nothing synchronises.
 * - Errors: argument errors found on the host return a non-zero tva_status and
 *   enqueue nothing.  Errors only visible on the device (a parent id out of range, a
 *   cu_* entry beyond the stated bounds, an internal wait that timed out) are
 *   written to *dev_status (an int32 the caller zeroes; the first error code wins)
 *   and the affected outputs are left unspecified.  Kernels never trap.
 */
#ifndef TVA_H_
#define TVA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TVA_OK = 0,
  TVA_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, bound exceeded */
  TVA_ERR_UNSUPPORTED = 2, /* head_dim or dtype this build does not implement      */
  TVA_ERR_BAD_TREE = 3,    /* parent[i] not in [-1, i)                              */
  TVA_ERR_WORKSPACE = 4,   /* workspace missing or smaller than tva_workspace_size  */
  TVA_ERR_CUDA = 5,        /* a CUDA runtime call failed (launch, attribute, ...)   */
  TVA_ERR_TIMEOUT = 6      /* an internal bounded wait expired (device status only) */
} tva_status;

typedef enum {
  TVA_BF16 = 0, /* bfloat16 inputs and output, fp32 accumulation */
  TVA_FP32 = 1, /* float32 inputs and output, fp32 accumulation  */
  TVA_FP16 = 2  /* float16 inputs and output, fp32 accumulation (LongSpec's own
                   precision, "Experiment details"); P is rounded to float16 */
} tva_dtype;

/* Problem description for the batched (varlen) entry points. */
typedef struct {
  int batch;          /* B >= 1                                                      */
  int num_q_heads;    /* Hq >= 1                                                     */
  int num_kv_heads;   /* Hkv >= 1, Hq % Hkv == 0                                     */
  int head_dim;       /* d: 64 or 128                                                */
  tva_dtype dtype;    /* q, k_cache, v_cache, tree_k, tree_v and out share it        */
  float softmax_scale;/* logit scale; 0 selects 1/sqrt(head_dim)                     */
  const int32_t* cu_prefix; /* device [B+1], cu_prefix[0] = 0, non-decreasing:
                               sequence b owns k_cache rows cu_prefix[b] ..
                               cu_prefix[b+1]-1                                       */
  const int32_t* cu_nodes;  /* device [B+1], cu_nodes[0] = 0, non-decreasing:
                               sequence b owns nodes (q/tree_k/tree_v/out rows and
                               parent entries) cu_nodes[b] .. cu_nodes[b+1]-1        */
  int max_prefix_len; /* host bound: every P_b <= max_prefix_len                     */
  int max_nodes;      /* host bound: every m_b <= max_nodes <= 128                   */
  int kv_capacity;    /* rows allocated in k_cache and v_cache (>= cu_prefix[B])     */
  int node_capacity;  /* rows allocated in q, tree_k, tree_v, out, lse, parent
                         (>= cu_nodes[B])                                            */
} tva_params;

/* Bytes of device workspace tree_verify_attn_varlen / _partials / _combine need for
 * `p` on the current device (it depends on the SM count).  Returns 0 when `p` is
 * invalid.  The workspace holds float32 partial outputs and log-sum-exps; it needs
 * no initialisation and its contents between the two stages are private. */
size_t tva_workspace_size(const tva_params* p);

/* Tree-verification attention over a ragged batch (LongSpec, "Fast Tree Attention").
 *   q        [N, Hq, d]    queries of the tree nodes (already projected/rotated)
 *   k_cache, v_cache [kv_capacity, Hkv, d]  cached prefix keys/values, ragged by
 *            cu_prefix (no mask applies to them)
 *   tree_k, tree_v   [N, Hkv, d]  keys/values of the tree nodes themselves
 *   parent   [N] int32     local parent ids per sequence (see conventions)
 *   out      [N, Hq, d]    attention output, same dtype as q
 *   lse      [N, Hq] float32  natural log of the sum of exp(scaled logits) over every
 *            key the row sees (prefix + ancestors + self)
 *   workspace, workspace_bytes  >= tva_workspace_size(p) bytes, 256-byte aligned
 *   dev_status  device int32, see conventions
 * Equivalent to tree_verify_attn_partials followed by tree_verify_attn_combine. */
tva_status tree_verify_attn_varlen(const tva_params* p, const void* q, const void* k_cache,
                                   const void* v_cache, const void* tree_k,
                                   const void* tree_v, const int32_t* parent, void* out,
                                   float* lse, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_status, void* stream);

/* Stage 1: attention partials.  Splits the prefix keys of every (sequence, KV head,
 * row group) into contiguous key ranges spread evenly over the GPU's SMs, adds the
 * tree keys (under the ancestor mask) as one more range, and writes each range's
 * output and log-sum-exp (the O_cache / O_specs, LSE_cache / LSE_specs of the
 * LongSpec aggregation) into `workspace`.  Arguments as for tree_verify_attn_varlen. */
tva_status tree_verify_attn_partials(const tva_params* p, const void* q, const void* k_cache,
                                     const void* v_cache, const void* tree_k,
                                     const void* tree_v, const int32_t* parent,
                                     void* workspace, size_t workspace_bytes,
                                     int32_t* dev_status, void* stream);

/* Stage 2: merges every row's partials with the log-sum-exp rule
 * LSE = log sum_s exp(LSE_s), out = sum_s O_s * exp(LSE_s - LSE)
 * (LongSpec, "Aggregation" and appendix Proposition) and writes out / lse.
 * `workspace` must hold the partials written by stage 1 for the same `p`. */
tva_status tree_verify_attn_combine(const tva_params* p, const void* workspace,
                                    size_t workspace_bytes, void* out, float* lse,
                                    int32_t* dev_status, void* stream);

/* Same computation as tree_verify_attn_varlen, for callers that cannot allocate
 * device memory (an engine that owns every allocation and forbids cudaMalloc on its
 * execution path, or a plugin interface with no workspace argument).  The paper has no
 * counterpart: this is a packaging of the same path.
 * Scratch: a fixed 32 MiB array compiled into the library and held on each GPU until
 * the process exits.  It is reserved when the module holding it is loaded on a device:
 * with CUDA's default lazy module loading that happens at this entry point's first
 * call on the device (with CUDA_MODULE_LOADING=EAGER, when the library's device code
 * is loaded), and that first call fails with TVA_ERR_CUDA (see tva_last_error()) if
 * the device has no 32 MiB left.  Problems whose tva_workspace_size() exceeds 32 MiB
 * are rejected with TVA_ERR_WORKSPACE (see tva_last_error()) before anything is
 * enqueued.  The first call on each device also looks the array's device address up
 * (cudaGetSymbolAddress), so make that first call before any stream capture.  Nothing
 * here calls an allocator.  All calls share the one array
 * and its contents carry over between calls (no step needs it zeroed); calls whose
 * work overlaps on the GPU (other streams, other host threads) race on it, so
 * serialise them.  Arguments otherwise as for tree_verify_attn_varlen. */
tva_status tree_verify_attn_varlen_noalloc(const tva_params* p, const void* q,
                                           const void* k_cache, const void* v_cache,
                                           const void* tree_k, const void* tree_v,
                                           const int32_t* parent, void* out, float* lse,
                                           int32_t* dev_status, void* stream);

/* Single-sequence convenience form (B = 1).  prefix_len and num_nodes are host
 * values; every other pointer is a device pointer laid out as above with B = 1.
 * The workspace and the cu_* arrays are library-owned: allocated on first use per
 * device (and grown when a larger problem arrives), released by tva_release().
 * Because it may allocate, do not call it for the first time inside stream capture.
 * Device-side errors go to a library-owned status word read by
 * tva_read_device_status().  Every call on a device shares that device's one
 * workspace: calls whose work overlaps on the GPU (several streams, several host
 * threads) race on it, so serialise them (the varlen forms take a caller-owned
 * workspace per call instead). */
tva_status tree_verify_attn(const void* q, const void* k_cache, const void* v_cache,
                            int prefix_len, const void* tree_k, const void* tree_v,
                            const int32_t* parent, int num_nodes, int num_q_heads,
                            int num_kv_heads, int head_dim, tva_dtype dtype, void* out,
                            float* lse, void* stream);

/* Copies the convenience form's device status into *host_status (a HOST pointer),
 * synchronising `stream`, and clears it.  TVA_OK when nothing was recorded. */
tva_status tva_read_device_status(int32_t* host_status, void* stream);

/* Frees the convenience form's library-owned buffers on every device. */
void tva_release(void);

/* Diagnostics, for testing the device-side timeout path; not for production use.
 * Sets, for this process and for launches made after the call, the limit of the
 * main-loop waits inside the tensor-core attention partials kernel (bf16 / fp16) in
 * nanoseconds (0 restores the default of 2 s).  With force_stall non-zero, that
 * kernel's MMA-issuing thread first waits on a barrier that nothing completes, so the
 * wait runs out: the kernel then raises its abort flag, lets every copy and MMA it
 * started finish (those drain waits always keep the 2 s limit), frees its tensor
 * memory, returns, and TVA_ERR_TIMEOUT is written to *dev_status.  Outputs of such a
 * launch are unspecified.  Call tva_diag_set_wait_limit(0, 0) to return to normal. */
void tva_diag_set_wait_limit(unsigned long long wait_limit_ns, int force_stall);

/* Diagnostics, for comparing two designs of the attention partials; not for production
 * use.  With enable non-zero, later calls whose problems have row groups of two M-tiles
 * (max_nodes * G > 128) at head_dim 128 in bf16 / fp16 run the CTA-pair partials kernel
 * (LongSpec's split key-value partials, "Fast Tree Attention", computed by two SMs per
 * worker: one M = 256 tensor-core MMA, cta_group::2, covers both M-tiles, each SM loads
 * half of every K/V tile) instead of the default one-SM-per-worker kernel.  Results
 * agree with the default within rounding-order differences (the row sums are added in
 * another order).  The pair kernel runs half as many workers, so a workspace sized while
 * it is selected can be too small for the default kernel (TVA_ERR_WORKSPACE).  Process-
 * wide; call with 0 to return to the default. */
void tva_diag_use_cta_pair(int enable);

/* Greedy longest accepted path per sequence ("Faster decoding", greedy contract).
 *   cu_nodes      [B+1] device, as in tva_params
 *   parent        [N] int32 local parent ids; draft_tok [N] int32 draft tokens
 *   target_argmax [N+B] int32: sequence b owns slots cu_nodes[b]+b ..
 *                 cu_nodes[b+1]+b; its slot 0 is the target's greedy token at the
 *                 prefix end and slot i+1 the target's greedy token after node i
 *   accept_len    [B] int32: nodes on the accepted path
 *   accept_path   [N] int32: per sequence, the accepted local ids root first, then -1
 *   next_token    [B] int32: slot[last+1] (slot[0] when nothing is accepted), the
 *                 correction or bonus token, so a cycle emits accept_len+1 tokens
 * Node i is accepted when it and every ancestor match (draft_tok[j] ==
 * slot[parent[j]+1]); the deepest accepted node wins and equal depths go to the
 * smaller local id.  Requires every m_b <= 128 and cu_nodes within node_capacity
 * (else TVA_ERR_INVALID_ARG in *dev_status for that sequence, whose accept_len and
 * next_token are then 0 and -1 and whose accept_path is left untouched). */
tva_status accept_longest_path(int batch, int node_capacity, const int32_t* cu_nodes,
                               const int32_t* parent,
                               const int32_t* draft_tok, const int32_t* target_argmax,
                               int32_t* accept_len, int32_t* accept_path,
                               int32_t* next_token, int32_t* dev_status, void* stream);

/* Commits each sequence's accepted path into the K/V cache ("Faster decoding", "The
 * scheduler must plan speculative work": after verification only the target KV of the
 * accepted draft prefix is committed and rejected branches are released).  The pages
 * give no interface; this one takes the acceptance walk's outputs as they are.
 *   batch, num_kv_heads, head_dim (64 or 128), dtype: as for the attention
 *   node_capacity rows in tree_k / tree_v [node_capacity, Hkv, d] (the tree nodes' K / V)
 *   max_nodes     bound on every m_b (<= 128; sizes the launch; a larger m_b is an
 *                 out-of-bounds sequence, see below)
 *   kv_capacity   rows in k_cache / v_cache [kv_capacity, Hkv, d]
 *   cu_nodes      [B+1] device, as in tva_params
 *   accept_len [B], accept_path [N]: as written by accept_longest_path
 *   dst_row       [B] device int32: first cache row for sequence b's committed rows
 *                 (for a cache whose sequences own reserved room after their prefix,
 *                 the prefix end)
 * Row j < accept_len[b] of the path (root first) is copied: K and V of tree row
 * cu_nodes[b] + accept_path[cu_nodes[b] + j] go to cache row dst_row[b] + j, bit for
 * bit.  No other cache row is written.  All pointers are device pointers; tree_k, tree_v,
 * k_cache and v_cache are 16-byte aligned and the sources must not overlap the
 * destination buffers (TVA_ERR_INVALID_ARG from the host, nothing launched).  A
 * sequence whose node range, path length, path ids or destination range is out of
 * bounds is left untouched and TVA_ERR_INVALID_ARG goes to *dev_status.  Ordered on
 * `stream` after the acceptance walk that wrote accept_len / accept_path. */
tva_status commit_accepted_kv(int batch, int num_kv_heads, int head_dim, tva_dtype dtype, int node_capacity,
                              int max_nodes, long long kv_capacity, const int32_t* cu_nodes,
                              const int32_t* accept_len, const int32_t* accept_path, const void* tree_k,
                              const void* tree_v, const int32_t* dst_row, void* k_cache, void* v_cache,
                              int32_t* dev_status, void* stream);

/* Stochastic verification of draft chains by modified rejection sampling ("Faster
 * decoding", "Modified rejection sampling keeps the target distribution"): left to
 * right, draft token x at a position is accepted with probability min(1, p(x)/q(x));
 * the first rejection ends the round with a correction token drawn from the residual
 * [p - q]_+ / Z; if all gamma drafts are accepted a bonus token is drawn from p at the
 * next position.  The pages give no interface; the random numbers are inputs.
 *   batch, vocab   B sequences over a vocabulary of V tokens
 *   max_draft      bound on every gamma_b (validated on the device)
 *   cu_draft       [B+1] device int32: sequence b's draft positions are
 *                  cu_draft[b] .. cu_draft[b+1]-1 (gamma_b of them)
 *   p              [p_rows, V] fp32 target probabilities; sequence b owns the gamma_b + 1
 *                  rows cu_draft[b] + b .. cu_draft[b+1] + b (the last is the bonus
 *                  position)
 *   q              [q_rows, V] fp32 draft probabilities, one row per draft position
 *   draft_tok      [sum gamma_b] int32, each drawn from its q row (q(x) > 0)
 *   u_accept       [sum gamma_b] fp32 uniforms in [0, 1), one per draft position
 *   u_sample       [B] fp32 uniforms in [0, 1), for the correction or bonus draw
 *   accept_len     [B] int32 out: drafts accepted
 *   out_token      [B] int32 out: the correction token (accept_len < gamma_b) or the
 *                  bonus token
 * Decisions: accept when p(x) >= q(x) or when u * q(x), rounded to fp32, is < p(x).
 * A draw is an inverse-CDF draw over masses quantised to 2^-40 and summed exactly as
 * integers (threshold floor(floor(u * 2^24) * Z / 2^24)), so it does not depend on the
 * order of the sums; an empty residual falls back to p.  p and q hold probabilities
 * (finite, >= 0); a negative or NaN entry is read as mass 0.  A sequence with bad bounds, a
 * token outside [0, V), q(x) = 0 or a uniform outside [0, 1) gets accept_len 0,
 * out_token -1 and TVA_ERR_INVALID_ARG in *dev_status. */
tva_status verify_chain_sampling(int batch, int vocab, int max_draft, long long p_rows, long long q_rows,
                                 const int32_t* cu_draft, const float* p, const float* q,
                                 const int32_t* draft_tok, const float* u_accept, const float* u_sample,
                                 int32_t* accept_len, int32_t* out_token, int32_t* dev_status, void* stream);

/* Tree verification for a Gated DeltaNet layer ("DFlash-TfM", Method 3, rollback-free
 * tree verification for GDN): the state update S_t = alpha_t (I - beta_t k_t k_t^T)
 * S_{t-1} + beta_t k_t v_t^T does not commute, so instead of an attention mask the tree
 * (topologically ordered) becomes one unit-lower-triangular system over its ancestor
 * pairs, solved by forward substitution, and the state itself is not updated (its
 * commit waits for the accepted branch).  Node i's output is o_i = S_i^T q_i with S_i
 * the state after running the update along the root-to-i path from S0.  The pages give
 * no interface.  All pointers are device pointers, row-major:
 *   batch, num_heads (H), head_dim (d: 64 or 128)
 *   dtype         type of q, k, v and out: TVA_FP32, or TVA_BF16 (the precision the page's
 *                 measurements use); beta, alpha and S0 are always fp32, and every
 *                 arithmetic step is fp32 (bf16 inputs widened, the output rounded once)
 *   node_capacity rows of q, k, v, out [node_capacity, H, d] and beta, alpha [node_capacity, H]
 *   max_nodes     bound on every m_b (<= 128)
 *   cu_nodes      [B+1], parent [N] local ids in [-1, i) (as for the attention)
 *   S0            [B, H, d, d] fp32 committed state at each sequence's prefix end (rows: keys)
 *   out           [N, H, d]
 * q, k, v, S0 and out are 16-byte aligned.  Any other dtype returns TVA_ERR_UNSUPPORTED.
 * A sequence outside the bounds is skipped with TVA_ERR_INVALID_ARG, a non-topological
 * parent array with TVA_ERR_BAD_TREE, in *dev_status. */
tva_status gdn_tree_verify(int batch, int num_heads, int head_dim, tva_dtype dtype, int node_capacity,
                           int max_nodes, const int32_t* cu_nodes, const int32_t* parent, const void* q,
                           const void* k, const void* v, const float* beta, const float* alpha, const float* S0,
                           void* out, int32_t* dev_status, void* stream);

/* Description of the last host-side CUDA or driver failure seen by this thread
 * (the call that failed and its error string), "" if none.  Thread-local storage,
 * valid until the thread's next failing call. */
const char* tva_last_error(void);

/* Human-readable name of a status code (static storage). */
const char* tva_status_string(tva_status s);

/* Number of workers (CTAs) the partials stage launches for `p` on the current
 * device, or -1 when `p` is invalid.  Informational. */
int tva_num_workers(const tva_params* p);

#ifdef __cplusplus
}
#endif

#endif /* TVA_H_ */
