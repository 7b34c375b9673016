/*
 * spec_verify.h -- C ABI of libspecverify: the data-parallel hot path of speculative decoding
 * on one NVIDIA GB300 (sm_103a).
 *
 * Three operations, each defined on the pages this library follows:
 *
 *   spec_verify_attn        Target-side verify attention.  The gamma+1 chain queries (the last
 *                           committed token plus gamma drafts), or the N nodes of a token tree,
 *                           attend over the full GQA KV cache of their sequence.
 *                           ("Guide to MagicDec", Solution section 2 and Implementation Step 3:
 *                           one target pass over prefix + drafts; "Speculative Decoding &
 *                           Medusa", section 4 and "Speculative Decoding in LLM Serving Systems",
 *                           Tree-based variants: tree attention where a node sees only its
 *                           ancestors.)
 *   spec_draft_window_attn  Draft-side single-query attention over a fixed-size ring-buffer
 *                           window of the last W tokens ("Guide to MagicDec", Solution section 1
 *                           and Implementation Step 1: bounded circular FIFO draft KV cache).
 *   spec_sample             The speculative-sampling step over the vocabulary: softmax of target
 *                           logits P and draft logits Q, left-to-right accept with probability
 *                           min(1, P(x)/Q(x)), residual resample from norm(max(P - Q, 0)) at the
 *                           first rejection, bonus token from P_{gamma+1} when all are accepted
 *                           ("Speculative Decoding & Medusa", section 2; "Speculative Decoding in
 *                           LLM Serving Systems", Accepting and rejecting); plus greedy chain and
 *                           greedy longest-accepted-path tree selection.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller, except the tree parent arrays,
 *    which are HOST pointers (the tree is small and shared by the batch; it is validated and
 *    turned into per-node ancestor bitmasks on the host before any launch).
 *  - Strides are in ELEMENTS.  The innermost dimension of every tensor is contiguous.
 *  - Calls are asynchronous on the given stream (a cudaStream_t; NULL = the legacy default
 *    stream).  They allocate no memory, keep no global mutable state and are thread-safe.
 *    Scratch memory is the caller's `workspace`, at least the size the matching *_workspace()
 *    query returns, 256-byte aligned.  Two calls that share a workspace must not overlap.
 *  - Host-side validation runs first and returns a negative status WITHOUT launching anything.
 *    A launch failure returns SPEC_ERR_CUDA.
 *  - Data errors that only the device can see (a kv_len or pos out of range, a token id outside
 *    [0, V)) never trap: the affected sequence's output is zeroed (attention) or its
 *    out_num_accepted is set to -1 (sampling), and a flag is OR-ed into the 32-bit status word
 *    at byte 0 of the workspace (SPEC_STATUS_*), which the call resets.  Read it with any
 *    device-to-host copy once the stream has reached the end of the call.
 *  - Device-side waits are bounded; a wait that runs out sets SPEC_STATUS_TIMEOUT and the kernel
 *    returns.
 */
#ifndef SPEC_VERIFY_H_
#define SPEC_VERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* spec_stream_t; /* same type as cudaStream_t */

/* return codes */
enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = -1, /* null pointer, bad size, stride, alignment or tree */
  SPEC_ERR_UNSUPPORTED = -2, /* a valid combination this build does not implement */
  SPEC_ERR_WORKSPACE = -3,   /* workspace missing, too small or misaligned */
  SPEC_ERR_CUDA = -4,        /* a CUDA runtime/driver call or kernel launch failed */
  SPEC_ERR_SCRATCH_LIMIT = -6 /* the problem needs more scratch than spec_verify_attn_noalloc has */
};

/* element types */
enum { SPEC_F32 = 0, SPEC_BF16 = 1 };

/* flags OR-ed into the device status word (byte 0 of the workspace) */
enum {
  SPEC_STATUS_BAD_KV_LEN = 1, /* kv_len[b] < nq or > Lmax: that sequence's output is zero   */
  SPEC_STATUS_BAD_POS = 2,    /* pos[b] < 1: that sequence's window output is zero           */
  SPEC_STATUS_BAD_TOKEN = 4,  /* a token id outside [0, V): that row's num_accepted is -1   */
  SPEC_STATUS_TIMEOUT = 8     /* a bounded device wait ran out; results are not valid        */
};

/* ------------------------------------------------------------------------------------------
 * spec_verify_attn
 *
 * For every sequence b, query row j in [0, nq) and query head h in [0, Hq):
 *     o[b, j, h, :] = softmax_t(scale * q[b, j, h, :] . k[b, g, t, :]) @ v[b, g, t, :]
 * with g = floor(h / (Hq / Hkv)) (contiguous GQA groups) and t over the keys row j sees.  The
 * cache of sequence b holds kv_len[b] entries, the last nq of which are the new query tokens
 * (already appended by the caller; Q and K already position-encoded):
 *   chain (tree_parent == NULL): row j sees keys 0 .. kv_len[b] - nq + j  (causal);
 *   tree  (tree_parent != NULL): node j sees the context keys [0, kv_len[b] - nq) and the tree
 *         keys kv_len[b] - nq + m for every m on the path from j to the root (m = j included).
 *
 * Layout (elements, innermost contiguous):
 *   q  [B, nq, Hq, D]   strides q_stride_b, q_stride_t, q_stride_h
 *   k,v[B, Hkv, Lmax, D] strides kv_stride_b, kv_stride_h; token stride = D
 *   o  [B, nq, Hq, D]   strides o_stride_b, o_stride_t, o_stride_h
 *   kv_len [B] int32 device
 * Types: kv_dtype SPEC_BF16 (q bf16) or SPEC_F32 (q f32); o_dtype SPEC_F32 or SPEC_BF16.
 * Fused append ("Speculative Decoding in LLM Serving Systems", the verify step appends the
 * drafts' K/V to the target cache; "Guide to MagicDec", Implementation Step 3): with k_new and
 * v_new set, the call first writes the nq new tokens' K/V rows
 *     k[b, g, kv_len[b] - nq + j, :] = k_new[b, j, g, :]   (and likewise v), j in [0, nq),
 * on the device, then attends over the updated cache; k and v are written through in that case
 * (the cache must be writable).  k_new, v_new: type kv_dtype, layout [B, nq, Hkv, D] with
 * strides new_stride_b, new_stride_t, new_stride_h (elements, innermost contiguous), owned by the
 * caller; k_new, v_new, k, v 16-byte aligned and all their strides multiples of 16 bytes (else
 * SPEC_ERR_INVALID_ARG).  A sequence whose kv_len is out of range gets no append (and is flagged
 * as below).
 * With k_new == v_new == NULL the caller has already written those rows.
 * Limits: D in {64, 128}; Hq % Hkv == 0; 1 <= B <= 4096; 1 <= nq; nq * (Hq/Hkv) <= 1024;
 *   tree: nq <= 64, tree_parent[0] == -1, 0 <= tree_parent[i] < i for i >= 1.
 *   bf16 K/V: base pointers 16-byte aligned, kv_stride_h and kv_stride_b multiples of 8.
 * scale == 0 selects 1/sqrt(D).
 * Accumulation is fp32 (scores, softmax, P.V); bf16 inputs are multiplied exactly.
 * debug_flags: 0 in normal use (any bit other than SPEC_DEBUG_NO_LOADS returns
 *   SPEC_ERR_INVALID_ARG).  SPEC_DEBUG_NO_LOADS is a test hook for the failure path of the bf16
 *   kernels: they issue no K/V copies, so the first bounded wait of every CTA runs out (after about
 *   one second), every kernel stops issuing, frees what it holds and returns, and the status word
 *   reads SPEC_STATUS_TIMEOUT; the output is not valid.  The fp32 kernel has no device waits and
 *   ignores the flag.
 * ---------------------------------------------------------------------------------------- */
enum { SPEC_DEBUG_NO_LOADS = 1 };

typedef struct spec_attn_args {
  int32_t B, Hq, Hkv, D, nq;
  int32_t q_dtype, kv_dtype, o_dtype;
  const void* q;
  int64_t q_stride_b, q_stride_t, q_stride_h;
  const void* k;
  const void* v;
  int64_t kv_stride_b, kv_stride_h;
  int32_t Lmax;
  int32_t reserved0;
  const int32_t* kv_len;      /* device [B] */
  const int32_t* tree_parent; /* HOST [nq], or NULL for chain verify */
  float scale;
  int32_t debug_flags;        /* 0, or SPEC_DEBUG_* test hooks (see below) */
  void* o;
  int64_t o_stride_b, o_stride_t, o_stride_h;
  void* workspace;
  size_t workspace_bytes;
  const void* k_new;          /* optional fused append (see above), device, or NULL */
  const void* v_new;
  int64_t new_stride_b, new_stride_t, new_stride_h;
} spec_attn_args;

/* Bytes of workspace spec_verify_attn needs for these sizes (host only, pure; reads no
 * pointer).  Returns 0 if the sizes are invalid. */
size_t spec_verify_attn_workspace(const spec_attn_args* args);
int spec_verify_attn(const spec_attn_args* args, spec_stream_t stream);

/* spec_verify_attn_noalloc -- the same verify attention with no caller workspace and no device
 * allocation anywhere.  The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory on their hot path (a serving engine that has handed all HBM to
 * its KV cache and weights up front, a plugin whose host framework owns every device
 * allocation, or a loop that cannot afford cudaMalloc/cudaFree, which synchronize the device).
 *
 * Scratch lives in one file-scope device array of SPEC_NOALLOC_SCRATCH_BYTES (64 MiB) that every
 * GPU which loads this library holds until the process exits.  args->workspace and
 * args->workspace_bytes are ignored.  A problem whose spec_verify_attn_workspace() size exceeds
 * the array returns SPEC_ERR_SCRATCH_LIMIT before anything is launched.
 *  - Every call looks up the array's device address in the calling thread's current context
 *    (cudaGetSymbolAddress); the first call in a context also loads the library's kernels into it,
 *    so make that first call before any stream capture.  Nothing is cached across contexts, so a
 *    caller may switch contexts (or reset the device) between calls.
 *  - Every call on a device shares the one array and leaves its contents behind; nothing in it
 *    has to start at zero (the per-call status word is cleared by the call itself).  Calls whose
 *    kernels overlap on the GPU (other streams, other host threads) race on the array: serialize
 *    them.  The status word (SPEC_STATUS_*) of the last call is at byte 0 of the array.
 * All other arguments, limits and results are those of spec_verify_attn. */
#define SPEC_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int spec_verify_attn_noalloc(const spec_attn_args* args, spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * spec_draft_window_attn
 *
 * Single-query draft attention over the draft's bounded window of W slots per sequence, kept as
 * a ring ([MagicDec] Implementation Step 1).  pos[b] counts the tokens written including the
 * current one.  With n_sinks = 0 token t (0-based) lives in slot t mod W and the visible tokens
 * are the last min(pos[b], W).  With n_sinks = S > 0 (attention sinks, [MagicDec] Best Practices
 * §1) the first S tokens keep slots 0..S-1 for good, token t >= S lives in slot
 * S + (t - S) mod (W - S), and the visible tokens are all of them while pos[b] <= W, else the S
 * first and the W - S most recent.  Either way the visible tokens fill slots 0..min(pos[b], W)-1
 * of the ring; since softmax over keys does not depend on their order, this equals attention over
 * the page's shift-left buffer.  If k_new/v_new are given, the current token's K/V take the slot
 * of token pos[b] - 1: the attention uses them in place of that slot's old contents, and the ring
 * is updated in place (the slot holds k_new/v_new once the call's work on the stream has
 * completed); k_new/v_new must not overlap the rings.
 *
 * Layout: q [B, Hq, D] (q_stride_b, q_stride_h); rings [B, Hkv, W, D] (ring_stride_b,
 * ring_stride_h; token stride D); k_new/v_new [B, Hkv, D] (new_stride_b, new_stride_h) or both
 * NULL; o [B, Hq, D] (o_stride_b, o_stride_h); pos [B] int32 device.
 * Types and limits as spec_verify_attn (nq = 1); W >= 1; 0 <= n_sinks < W (else
 * SPEC_ERR_INVALID_ARG).
 * Workspace: spec_draft_window_attn_workspace() bytes, status word at byte 0, cleared by the call.
 *   For bf16 rings with up to 16 query rows per kv head the kernel clears it itself (no separate
 *   memset on the stream) and tags workspace bytes 8-15 with its launch.
 * ---------------------------------------------------------------------------------------- */
typedef struct spec_window_args {
  int32_t B, Hq, Hkv, D, W;
  int32_t q_dtype, kv_dtype, o_dtype;
  const void* q;
  int64_t q_stride_b, q_stride_h;
  void* k_ring;
  void* v_ring;
  int64_t ring_stride_b, ring_stride_h;
  const int32_t* pos; /* device [B] */
  const void* k_new;  /* device [B, Hkv, D] or NULL */
  const void* v_new;
  int64_t new_stride_b, new_stride_h;
  float scale;
  int32_t n_sinks;    /* attention-sink slots at the front of the ring (0: plain ring) */
  void* o;
  int64_t o_stride_b, o_stride_h;
  void* workspace;
  size_t workspace_bytes;
} spec_window_args;

size_t spec_draft_window_attn_workspace(const spec_window_args* args);
int spec_draft_window_attn(const spec_window_args* args, spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * spec_sample
 *
 * SPEC_SAMPLE_CHAIN (stochastic, temperature 1, n = gamma >= 1):
 *   P_i = softmax(target_logits[b, i]), Q_i = softmax(draft_logits[b, i]).  For i = 1..gamma
 *   accept x_i = draft_tokens[b, i-1] iff u_i * Q_i(x_i) < P_i(x_i) (u_i = uniforms[b, i-1]),
 *   stopping at the first rejection (k accepted).  Then draw y by inverse CDF in token-id order
 *   with u_{gamma+1} = uniforms[b, gamma] from r = max(P_{k+1} - Q_{k+1}, 0) if k < gamma, else
 *   r = P_{gamma+1}: y = min{y : sum_{z<=y} r_z > u_{gamma+1} * sum r} (if sum r == 0, r = P_{k+1};
 *   if no index qualifies through rounding, the largest y with r_y > 0).
 *   Output: out_tokens[b, 0..k] = x_1..x_k, y; the rest of the row -1; out_num_accepted[b] = k.
 * SPEC_SAMPLE_CHAIN_GREEDY (n = gamma >= 0): x_i accepted while it equals argmax P_i (ties to the
 *   smallest id, so a row of all -inf gives id 0); then the argmax of row k+1 is emitted.
 *   draft_logits and uniforms unused.
 * SPEC_SAMPLE_TREE_GREEDY (n = N nodes, tree_parent HOST [N]): row i of target_logits holds the
 *   logits after node i; node i >= 1 is accepted iff its parent is accepted and
 *   draft_tokens[b, i] (the node's token) equals the argmax of its parent's row; node 0 (the last
 *   committed token) is accepted.  The deepest accepted node d (ties to the smallest index) is
 *   chosen: out_tokens = tokens of the path's nodes at depth 1..depth(d), then argmax of row d;
 *   out_path_nodes (optional) = those node ids; out_num_accepted = depth(d).
 * SPEC_SAMPLE_TREE (stochastic tree, n = N nodes, tree_parent HOST [N]): multi-step speculative
 *   sampling -- the chain test applied to a node's children in turn (the pages name SpecInfer's
 *   tree verification, "Speculative Decoding in LLM Serving Systems", without its rule; this is
 *   the reading used).  Row n of target_logits is the target after node n (P_n), row n of
 *   draft_logits the distribution node n's children were drawn from (Q_n; rows of leaves are not
 *   read); uniforms [B, N].  From node n = 0: R = P_n; for each child c of n in increasing index
 *   order accept iff uniforms[b, c] * Q_n(x_c) < R(x_c) (x_c = draft_tokens[b, c]) and continue
 *   at c, else R = max(R - Q_n, 0) normalised (R = P_n if that has no mass) and test the next
 *   child.  When no child is accepted, y is drawn from R by inverse CDF with uniforms[b, 0] as in
 *   the chain mode.  Outputs as in SPEC_SAMPLE_TREE_GREEDY (path tokens, then y).
 *
 * Layout: logits rows are V contiguous fp32; target_logits [B, rows_t, V] with batch stride
 *   tl_stride_b (rows_t = gamma+1 chain, N tree); draft_logits [B, gamma, V] or [B, N, V]
 *   (dl_stride_b); draft_tokens [B, gamma] or [B, N] int32 (tok_stride_b); uniforms [B, gamma+1]
 *   or [B, N] fp32 in [0, 1)
 *   (u_stride_b); out_tokens / out_path_nodes [B, out_cols] int32 (row stride out_cols);
 *   out_num_accepted [B] int32.
 * Limits: V % 4 == 0, logits pointers 16-byte aligned and tl/dl strides multiples of 4;
 *   1 <= B; chain: 1 <= gamma <= 32 (stochastic), 0 <= gamma <= 32 (greedy),
 *   out_cols >= gamma + 1; tree: 1 <= N <= 64, out_cols >= max depth + 1.
 *   Logits hold no NaN, and in the stochastic modes every row the rule reads holds a value above
 *   -inf (a softmax needs one); otherwise the outputs (tokens, counts, paths) are unspecified,
 *   though the kernels still touch no memory outside the call's buffers.  -inf entries are
 *   allowed.
 * Floating point: V > 2048 (the statistics + finish kernels) uses no fp64 at all.  Each thread
 *   sums its own elements in fp32 (pairwise or compensated); every sum above that -- across lanes,
 *   warps, CTAs and the cluster -- is float-float (Knuth's TwoSum, about 44 significant bits), in a
 *   fixed order, with no floating-point atomics, so every decision is reproducible.  The terms of
 *   the softmax normalisers and of the residual CDF are fp32 2^x of the max-subtracted, log2(e)-
 *   scaled logit (relative error about 2^-22).  The accept ratio P(x)/Q(x) is
 *   exp((t_x - M_t) - (d_x - M_d)) * Z_d / Z_t with the exponent formed exactly as a float-float
 *   and evaluated by fp32 expf, then fp32 division (relative error a few 1e-7).
 *   V <= 2048 (one warp per sequence): fp32 exponentials, fp64 sums and fp64 accept ratios.
 *   Either way a decision can differ from exact arithmetic only when its exact value lies within
 *   about 1e-6 (relative) of its threshold.
 * Diagnostics: after a SPEC_SAMPLE_CHAIN call with V > 2048, the 32-bit word at byte 4 of the
 *   workspace holds the launch shape of the accept/draw kernel: the number of CTAs that share one
 *   sequence's vocabulary (a thread-block cluster) in the low byte, and bit 8 set when the draw
 *   re-reads the residual row from memory instead of scanning values kept on chip.  No result
 *   depends on it; tests read it to know which code path a shape exercised.
 * Status: the status word at byte 0 of the workspace is cleared by the call; with V > 2048 (chain
 *   and greedy modes) the first kernel clears it itself (no separate memset on the stream) and
 *   tags workspace bytes 8-15 with its launch.
 * ---------------------------------------------------------------------------------------- */
enum { SPEC_SAMPLE_CHAIN = 0, SPEC_SAMPLE_CHAIN_GREEDY = 1, SPEC_SAMPLE_TREE_GREEDY = 2, SPEC_SAMPLE_TREE = 3 };

typedef struct spec_sample_args {
  int32_t mode, B, n, V;
  const float* target_logits;
  int64_t tl_stride_b;
  const float* draft_logits;
  int64_t dl_stride_b;
  const int32_t* draft_tokens;
  int64_t tok_stride_b;
  const int32_t* tree_parent; /* HOST [N] (tree mode) */
  const float* uniforms;
  int64_t u_stride_b;
  int32_t out_cols;
  int32_t reserved0;
  int32_t* out_tokens;
  int32_t* out_num_accepted;
  int32_t* out_path_nodes; /* tree mode, optional */
  void* workspace;
  size_t workspace_bytes;
} spec_sample_args;

size_t spec_sample_workspace(const spec_sample_args* args);
int spec_sample(const spec_sample_args* args, spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * spec_lmhead_sample -- the LM-head projection fused with verification
 *
 * The verified rows' logits are the target's final hidden states times the LM-head (unembedding)
 * matrix ("Speculative Decoding in LLM Serving Systems", The algorithm: one target pass gives a
 * next-token distribution per drafted position; "Guide to MagicDec", Implementation Step 3).
 * Greedy modes only need each row's argmax, so they never write the logits: a tcgen05 GEMM reduces
 * its fp32 accumulators straight to one running (max, argmax) key per row, and the rule of
 *   SPEC_SAMPLE_CHAIN_GREEDY (n = gamma: rows 0..gamma, draft_tokens [B, gamma]) or
 *   SPEC_SAMPLE_TREE_GREEDY  (n = N nodes: rows 0..N-1, node tokens [B, N], tree_parent HOST [N])
 * is applied to the argmaxes exactly as spec_sample does (ties to the smaller token id).
 * Stochastic modes need whole normalised rows (the residual draw), so the same GEMM writes the fp32
 * target logits [B, R, V] -- into out_logits if given, else into the workspace, where at these
 * sizes (20 MB for 40 rows of a 128K vocabulary) they are read back from L2 -- and the
 * speculative-sampling kernels of spec_sample then run on them in the same call:
 *   SPEC_SAMPLE_CHAIN (n = gamma >= 1: rows 0..gamma, draft_logits [B, gamma, V], uniforms
 *                      [B, gamma + 1]) and
 *   SPEC_SAMPLE_TREE  (n = N nodes: draft_logits [B, N, V], uniforms [B, N], tree_parent HOST [N]),
 * with exactly the rules, outputs and numerics of spec_sample in that mode.
 *
 * Layout: hidden bf16 [B, R, d] contiguous (R = gamma + 1 or N), weight bf16 [V, d] contiguous,
 *   both 16-byte aligned; draft_tokens int32 with batch stride tok_stride_b; out_tokens /
 *   out_path_nodes [B, out_cols], out_num_accepted [B] as for spec_sample.  Stochastic modes:
 *   draft_logits fp32 with batch stride dl_stride_b (rows of V contiguous), uniforms fp32 with
 *   batch stride u_stride_b, out_logits (optional) fp32 [B, R, V] contiguous, all 16-byte aligned.
 * Limits: d a multiple of 64 (up to 65 536); 1 <= V <= 2^24 (stochastic: V % 4 == 0 and
 *   V <= 2^20); B * R <= 256; tree: N <= 64, out_cols >= max depth + 1; chain: 0 <= gamma <= 32
 *   (stochastic: >= 1), out_cols >= gamma + 1.
 * Floating point: bf16 products accumulated in fp32 on the tensor cores; greedy argmaxes compare
 *   those fp32 values (an exact tie goes to the smaller id; two logits within the fp32 rounding of
 *   a d-term sum of each other may come out in either order); stochastic modes sample from those
 *   fp32 logits as spec_sample does.
 * Workspace: spec_lmhead_sample_workspace() bytes (the status word at byte 0, the row keys or the
 *   logits and the sampling workspace), 256-byte aligned.
 * ---------------------------------------------------------------------------------------- */
typedef struct spec_lmhead_args {
  int32_t mode, B, n, d, V;
  int32_t out_cols;
  const void* hidden;          /* bf16 [B, R, d], device */
  const void* weight;          /* bf16 [V, d], device */
  const int32_t* draft_tokens; /* device */
  int64_t tok_stride_b;
  const int32_t* tree_parent;  /* HOST [N] (tree modes) */
  int32_t* out_tokens;
  int32_t* out_num_accepted;
  int32_t* out_path_nodes;     /* tree modes, optional */
  void* workspace;
  size_t workspace_bytes;
  /* stochastic modes only (NULL / 0 in greedy modes) */
  const float* draft_logits;   /* device [B, gamma | N, V] */
  int64_t dl_stride_b;
  const float* uniforms;       /* device [B, gamma + 1 | N] */
  int64_t u_stride_b;
  float* out_logits;           /* device [B, R, V], optional: the projected target logits */
} spec_lmhead_args;

size_t spec_lmhead_sample_workspace(const spec_lmhead_args* args);
int spec_lmhead_sample(const spec_lmhead_args* args, spec_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * spec_commit
 *
 * The rollback step after verification ("Speculative Decoding in LLM Serving Systems", Accepting
 * and rejecting; "Guide to MagicDec", Implementation Step 3; "Speculative Decoding & Medusa" §4):
 * keep the K/V of the accepted tokens and drop the rest, on the device, from spec_sample's
 * outputs, so that no host round trip sits between rounds.  The nq positions verified in the
 * round are the last nq of each sequence's cache, kv_len[b] - nq .. kv_len[b] - 1.
 *
 * SPEC_COMMIT_CHAIN (nq = gamma + 1): position kv_len - nq holds the last committed token and the
 *   next gamma the drafts; with k = num_accepted[b] the first k + 1 stay:
 *   kv_len[b] = kv_len[b] - nq + 1 + k.  No K/V moves (k and v may be NULL).
 * SPEC_COMMIT_TREE (nq = N nodes, N <= 64): node i sits at position kv_len - N + i, node 0 (the
 *   root) being the last committed token; with the accepted path path_nodes[b, 0..k-1] (depths
 *   1..k, as spec_sample's out_path_nodes reports it) the K/V of path node j move to position
 *   kv_len - N + 1 + j, for every kv head, and kv_len[b] = kv_len[b] - N + 1 + k.
 *
 * A sequence with num_accepted outside [0, nq - 1] (tree: or above path_cols), kv_len outside
 * [nq, Lmax] or (tree) a path node outside [1, N) is left unchanged and SPEC_STATUS_BAD_TOKEN /
 * SPEC_STATUS_BAD_KV_LEN is set in the status word (byte 0 of the workspace).
 *
 * Layout: k, v [B, Hkv, Lmax, D] with strides as spec_verify_attn (kv_dtype SPEC_BF16 or
 * SPEC_F32, 4-byte aligned, strides even for bf16); kv_len [B] int32 device, read and written;
 * num_accepted [B] int32 device; path_nodes [B, path_cols] int32 device, path_stride_b >=
 * path_cols elements between rows (tree only; spec_sample's out_path_nodes fits as it is).  workspace: spec_commit_workspace() bytes, 256-byte aligned.
 * ---------------------------------------------------------------------------------------- */
typedef enum { SPEC_COMMIT_CHAIN = 0, SPEC_COMMIT_TREE = 1 } spec_commit_mode;

typedef struct spec_commit_args {
  int32_t mode, B, Hkv, D, nq, Lmax;
  int32_t kv_dtype, path_cols; /* tree: node ids per path row (>= the largest num_accepted) */
  void* k; /* device, tree mode */
  void* v;
  int64_t kv_stride_b, kv_stride_h;
  int32_t* kv_len;             /* device [B], in/out */
  const int32_t* num_accepted; /* device [B] */
  const int32_t* path_nodes;   /* device [B, path_stride_b], tree mode */
  int64_t path_stride_b;
  void* workspace;
  size_t workspace_bytes;
} spec_commit_args;

size_t spec_commit_workspace(const spec_commit_args* args);
int spec_commit(const spec_commit_args* args, spec_stream_t stream);

/* Text for a return code. */
const char* spec_status_string(int status);
/* ABI version: bump on any struct or semantic change. */
int spec_abi_version(void);
/* sizeof() of the argument structs as compiled into the library, so that a binding can check
 * its own layout: which = 0 spec_attn_args, 1 spec_window_args, 2 spec_sample_args,
 * 3 spec_commit_args, 4 spec_lmhead_args; else 0. */
size_t spec_abi_struct_size(int which);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H_ */
