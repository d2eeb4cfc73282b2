/*
 * tv.h -- C ABI of the tree speculative-decoding verify step (libtv.so).
 *
 * One verify step scores a flattened draft tree of N nodes against each
 * sequence's paged KV cache in a single pass, reduces each node's target
 * logits to an argmax, walks the tree greedily on the GPU and commits the
 * accepted nodes' K/V into the cache.  The five calls below are that step, in
 * order:
 *
 *   tv_build_ancestors -> tv_tree_attention -> tv_argmax -> tv_tree_walk -> tv_commit_kv
 *
 * Source pages (cited by title and section):
 *   [SPEC]   "Tree spec-decode -> vLLM serve integration spec": "What's proven",
 *            "2. Verify: tree attention mask", "3. Rejection sampler: tree
 *            walk", "Layout contract".
 *   [DDTREE] "From Linear to Tree-Walk: Validating DDTree's Core Algorithm in
 *            vLLM": "The Successful Test".
 *
 * Conventions shared by every call
 *   - Every pointer argument is DEVICE memory owned by the caller (for example
 *     allocated by PyTorch).  The library allocates nothing and keeps no
 *     pointer after the call returns, with one exception: tv_argmax_noalloc
 *     keeps its partials in a fixed static device array of the library and
 *     caches that array's device address per device (see its comment).
 *   - Every call only enqueues work on `stream` (a cudaStream_t; NULL means the
 *     legacy default stream) and never synchronises with the host.
 *   - Stream order holds as usual.  Some kernels are launched as programmatic
 *     dependents (tv_tree_attention, tv_tree_walk, tv_commit_kv and the merge
 *     kernels of tv_argmax and tv_topk): they may become resident while the
 *     kernel before them is still running, but only when that kernel is one of
 *     this library's that releases its dependents early, and they read what
 *     that kernel writes only after it has completed.  tv_tree_attention reads
 *     q, the context lengths, the tree K/V, the KV cache and the block table
 *     early; none of this library's kernels that release their dependents
 *     early writes any of those (tv_commit_kv, which writes the cache and the
 *     context lengths, releases nothing early), and a caller's own kernel
 *     releases nothing early, so stream order applies.  tv_tree_attention's
 *     own grids release their dependents early too, so its `out` must not be
 *     the `q` of a tv_tree_attention call enqueued directly after it: a
 *     caller's kernel between the two (as a model's projection is) restores
 *     plain stream order.
 *   - The return value reports argument/shape validation and launch errors
 *     only.  Data errors found on the device (a malformed tree, a bad block id)
 *     are written to the per-sequence `status` array (int32 [B]): 0 = ok, else a
 *     tv_status code.  tv_build_ancestors writes status[b] for every b; later
 *     calls only ever write a non-zero code into it.  Kernels never trap, never
 *     print and never loop without bound.
 *   - bf16 means the 16-bit brain float format; "int32 [B, N]" means a dense
 *     row-major array.
 *
 * Tree layout ([SPEC] "Layout contract"): tokens[N], parent[N], depth[N] per
 * sequence.  parent[t] is the index of t's parent node, -1 when t is a child of
 * the last accepted token.  Parents precede children (parent[t] < t), and
 * depth[t] = 1 when parent[t] = -1, else depth[parent[t]] + 1.  N <= 64.
 */
#ifndef TV_H_
#define TV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int tv_status;
#define TV_OK 0
#define TV_ERR_ARG 1          /* bad pointer, size or shape (host check)         */
#define TV_ERR_TREE 2         /* malformed parent[] / depth[] (device check)      */
#define TV_ERR_BLOCK 3        /* block id or block-table slot out of range        */
#define TV_ERR_CUDA 4         /* a CUDA launch or driver call failed              */
#define TV_ERR_UNSUPPORTED 5  /* valid but not supported shape or dtype           */
#define TV_ERR_SCRATCH_LIMIT 6 /* too large for a no-allocation entry point's fixed scratch */

#define TV_F32 0
#define TV_BF16 1

#define TV_BLOCK_SIZE 16      /* paged-KV block size (tokens) */
#define TV_MAX_NODES 64

typedef void *tv_stream;      /* a cudaStream_t */

/* Human-readable name of a status code (static string, never NULL). */
const char *tv_status_string(tv_status s);

/*
 * tv_build_ancestors -- ancestor bitmask and position ids of every tree node.
 * [SPEC] "2. Verify": node t attends node a iff a is an ancestor of t or t
 * itself; position_ids[t] = ctx_len - 1 + depth(t).
 *
 *   parent, depth  int32 [B, N]   tree layout (see above)
 *   ctx_len        int32 [B]      tokens already in the cache, including the
 *                                 last accepted token
 *   anc            uint64 [B, N]  out: bit a of anc[b][t] set iff node a is an
 *                                 ancestor-or-self of node t
 *   pos            int32 [B, N]   out: ctx_len[b] - 1 + depth[b][t]
 *   status         int32 [B]      out: 0, or TV_ERR_TREE when some parent[t] is
 *                                 outside [-1, t-1] or some depth disagrees with
 *                                 the parent chain.  For such a sequence anc and
 *                                 pos hold in-range but unspecified values and
 *                                 the walk accepts nothing.
 * Errors: TV_ERR_ARG for NULL pointers, B < 0, N < 0 or N > 64.
 * B = 0 or N = 0 launches nothing (status is still written when B > 0).
 */
tv_status tv_build_ancestors(const int32_t *parent, const int32_t *depth,
                             const int32_t *ctx_len, int B, int N, uint64_t *anc,
                             int32_t *pos, int32_t *status, tv_stream stream);

/*
 * Arguments of tv_tree_attention.
 * [SPEC] "2. Verify": every node attends (a) the whole paged-KV context of its
 * sequence and (b) its tree ancestors and itself; the mask composes with the
 * layer's sliding window (left, right).
 *
 *   q          bf16 [B, N, Hq, D]         node queries (post-RoPE)
 *   k_tree     bf16 [B, N, Hkv, D]        node keys / values (post-RoPE)
 *   v_tree     bf16 [B, N, Hkv, D]
 *   k_cache    bf16 [num_blocks, Hkv, 16, D]   paged context cache
 *   v_cache    bf16 [num_blocks, Hkv, 16, D]
 *   block_table int32 [B, max_blocks]     context key j of sequence b lives in
 *                                         block block_table[b][j/16], row j%16
 *   ctx_len    int32 [B]                  context keys 0 .. ctx_len-1 are read
 *   pos, anc   from tv_build_ancestors
 *   window_left  keys at positions >= pos[t] - window_left are visible;
 *                -1 = no window (global attention)
 *   window_right must be -1 or >= 0; every visible key precedes or equals the
 *                query position, so the right bound never removes a key
 *   sm_scale   softmax scale on q.k; 0 means 1/sqrt(D)
 *   num_splits context splits per (sequence, KV head) of the CUDA-core
 *              kernel and of the D = 256 tensor-core kernel; 0 = chosen by the
 *              library (the D = 128 tensor-core kernel balances its work itself
 *              and ignores it)
 *   kernel     0 = automatic (tensor cores when the shape allows, else CUDA
 *              cores), 1 = CUDA-core kernel, 2 = tensor-core kernel
 *              (TV_ERR_UNSUPPORTED outside its shapes: D = 128 with
 *              (Hq/Hkv)*N <= 128 and B <= 1024, or D = 256 with
 *              (Hq/Hkv)*N <= 128)
 *   max_ctas   at most this many persistent CTAs for the D = 128 tensor-core
 *              kernel, one per SM (0 = every SM).  Leaving SMs free lets
 *              another kernel that does not depend on this one, such as
 *              tv_argmax_sm on a second stream, run beside it.  Ignored by the
 *              other kernels.
 *   out        bf16 [B, N, Hq, D]         softmax(scale q.K^T) V per node and head
 *   status     int32 [B]                  TV_ERR_BLOCK is recorded when a needed
 *                                         block id is outside [0, num_blocks) or
 *                                         ctx_len exceeds max_blocks*16 (that
 *                                         sequence's outputs are then
 *                                         unspecified but finite); TV_ERR_CUDA
 *                                         when a pipeline wait timed out
 * Query head h reads KV head h / (Hq / Hkv).  Supported: D in {64, 128, 256},
 * Hq % Hkv == 0, block_size == 16, N <= 64, (Hq/Hkv)*N <= 256.
 */
typedef struct tv_attn_args {
  const void *q;
  const void *k_tree;
  const void *v_tree;
  const void *k_cache;
  const void *v_cache;
  const int32_t *block_table;
  const int32_t *ctx_len;
  const int32_t *pos;
  const uint64_t *anc;
  int B, N, Hq, Hkv, D;
  int block_size;
  int max_blocks;
  int num_blocks;
  int window_left;
  int window_right;
  float sm_scale;
  int num_splits;
  int kernel;
  int max_ctas;
  void *out;
  int32_t *status;
} tv_attn_args;

/*
 * Bytes of scratch tv_tree_attention needs for these arguments (fp32 split
 * partials; 0 when one split suffices).  Only the shape fields, num_splits and
 * window_left are read.
 */
size_t tv_tree_attention_workspace_size(const tv_attn_args *a);

/*
 * tv_tree_attention -- masked tree attention over the paged context plus the
 * node -> node ancestor block, fp32 accumulation, bf16 output.
 * `workspace` is device memory of at least tv_tree_attention_workspace_size(a)
 * bytes, 256-byte aligned (may be NULL when that size is 0).
 * Errors: TV_ERR_ARG (NULL pointer, inconsistent sizes, small workspace),
 * TV_ERR_UNSUPPORTED (D, block size or group size outside the supported set).
 */
tv_status tv_tree_attention(const tv_attn_args *a, void *workspace,
                            size_t workspace_bytes, tv_stream stream);

/*
 * Bytes of scratch tv_argmax needs for `rows` rows of `V` logits of `dtype`:
 * room for the (value, index) partials of rows that are cut between thread
 * blocks, whichever plan the call takes (0 when no plan cuts a row).
 */
size_t tv_argmax_workspace_size(int64_t rows, int64_t V, int dtype);

/*
 * tv_argmax -- index of the maximum of every logits row.
 * [SPEC] "3. Rejection sampler": the walk consumes argmax(target_logits[t]).
 *
 *   logits     dtype [rows, row_stride] (TV_BF16 or TV_F32), first V used
 *   out_idx    int32 [rows]   min { i : x[i] == max_j x[j] }: ties go to the
 *                             lowest index, +0 == -0, a NaN counts as -inf
 *                             (a row of NaN / -inf only gives 0)
 *   workspace  >= tv_argmax_workspace_size(rows, V, dtype) bytes, 16-aligned
 * Dense rows (row_stride == V, 16-byte aligned base, V * element size a
 * multiple of 16) with at least 32 KiB of logits per SM are streamed in equal
 * contiguous ranges, one per warp of a one-block-per-SM grid; other inputs
 * take one thread block per row chunk.  Both give the same indices.
 * Errors: TV_ERR_ARG (NULL pointers, V < 1, row_stride < V, rows or V beyond
 * int32 indexing, small workspace), TV_ERR_UNSUPPORTED (other dtypes),
 * TV_ERR_CUDA (launch failure).
 */
tv_status tv_argmax(const void *logits, int dtype, int64_t rows, int64_t V,
                    int64_t row_stride, int32_t *out_idx, void *workspace,
                    size_t workspace_bytes, tv_stream stream);

/*
 * tv_argmax_sm -- tv_argmax with its streaming plan held to at most sm_limit
 * SMs (one CTA each; 0 = every SM), so that it can run beside a kernel that
 * occupies the other SMs, e.g. tv_tree_attention with max_ctas = SMs -
 * sm_limit on another stream: the two read HBM at the same time.  The chunk
 * plan ignores the limit.  Same arguments, workspace, result and errors as
 * tv_argmax otherwise (tv_argmax_workspace_size covers every limit).
 */
tv_status tv_argmax_sm(const void *logits, int dtype, int64_t rows, int64_t V,
                       int64_t row_stride, int32_t *out_idx, void *workspace,
                       size_t workspace_bytes, int sm_limit, tv_stream stream);

/*
 * tv_argmax_noalloc -- tv_argmax for callers that cannot allocate device memory.
 * The verify-step pages have no counterpart to this call; it exists for the
 * library's users.  Some callers may not call cudaMalloc at all while they
 * run: a serving loop whose device memory is all owned by one pool allocator,
 * a plugin host that hands a kernel only its input and output buffers, or a
 * latency-critical decode loop in which cudaMalloc (which can synchronise the
 * device) is not allowed.  Such callers cannot provide tv_argmax's workspace.
 *
 * Same arguments, result and errors as tv_argmax, minus the workspace.  The
 * split partials live in one fixed array of 8192 (value, index) pairs
 * (64 KiB) in the library's static device memory, which every GPU that loads
 * the library keeps until the process exits.  A shape whose plan needs more
 * pairs than that returns TV_ERR_SCRATCH_LIMIT and launches nothing (on a
 * 152-SM GPU no shape needs more than 4,864: two per warp of the streaming
 * plan).  The call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 *
 * The first call made with a given device current looks up the array's device
 * address (cudaGetSymbolAddress) and caches it; make that first call before
 * any stream capture.  The cached address belongs to the device's primary
 * context: after cudaDeviceReset (or any other teardown of that context) it is
 * stale, so this call must not be used again in that process.  Every call shares the one array and leaves its partials
 * behind (each call writes every partial it reads, so nothing needs clearing),
 * so calls that may overlap on the GPU -- on different streams without
 * ordering between them -- race and must not be issued.
 */
tv_status tv_argmax_noalloc(const void *logits, int dtype, int64_t rows, int64_t V,
                            int64_t row_stride, int32_t *out_idx, tv_stream stream);

/*
 * tv_tree_walk -- greedy acceptance walk over the tree, on the GPU.
 * [SPEC] "What's proven" and "3. Rejection sampler": from the root, follow the
 * child whose token equals the target argmax of the current node, emit it and
 * repeat; finally emit the last argmax (the bonus token).  The accepted tokens
 * then equal plain greedy decoding of the target, for any tree.
 *
 *   tokens, parent int32 [B, N]  tree layout
 *   argmax         int32 [B, N]  target argmax of every node (tv_argmax)
 *   root_pred      int32 [B]     target argmax at the last accepted token (the
 *                                previous step's bonus token)
 *   status         int32 [B]     in: a non-zero entry makes that sequence
 *                                accept nothing (n_acc = 0, emit root_pred)
 *   out_tokens     int32 [B, N+1] out: emitted tokens, -1 past n_emit
 *   n_emit         int32 [B]     out: n_acc + 1
 *   acc_nodes      int32 [B, N]  out: accepted node ids root-first, -1 past n_acc
 *   n_acc          int32 [B]     out: accepted tree nodes
 * When several children of the current node carry the predicted token the
 * lowest node index is followed.  The loop runs at most N steps.
 * Errors: TV_ERR_ARG (NULL pointers, B < 0, N outside [0, 64]).
 */
tv_status tv_tree_walk(const int32_t *tokens, const int32_t *parent,
                       const int32_t *argmax, const int32_t *root_pred,
                       const int32_t *status, int B, int N, int32_t *out_tokens,
                       int32_t *n_emit, int32_t *acc_nodes, int32_t *n_acc,
                       tv_stream stream);

/*
 * tv_commit_kv -- write the accepted nodes' K/V rows into the paged cache.
 * [SPEC] "3. Rejection sampler": the accepted tokens and their KV are kept,
 * rejected branches are discarded.  The i-th accepted node (depth i+1) is
 * written at position p = ctx_len_in[b] + i, i.e. cache block
 * block_table[b][p/16], row p%16, for every KV head.  Nothing else is written.
 *
 *   k_tree, v_tree  bf16 [B, N, Hkv, D]
 *   acc_nodes, n_acc from tv_tree_walk (read on the device: no host sync)
 *   ctx_len_in      int32 [B]
 *   block_table     int32 [B, max_blocks]
 *   k_cache, v_cache bf16 [num_blocks, Hkv, 16, D]  updated in place
 *   ctx_len_out     int32 [B]  out: ctx_len_in + n_acc (ctx_len_in when the
 *                              sequence's commit fails); a separate array so a
 *                              step can be replayed
 *   status          int32 [B]  TV_ERR_BLOCK when a needed slot is beyond
 *                              max_blocks or a block id is outside
 *                              [0, num_blocks): that sequence commits nothing
 * Errors: TV_ERR_ARG (NULL pointers, bad sizes), TV_ERR_UNSUPPORTED (D not a
 * multiple of 8).
 */
tv_status tv_commit_kv(const void *k_tree, const void *v_tree, const int32_t *acc_nodes,
                       const int32_t *n_acc, const int32_t *ctx_len_in,
                       const int32_t *block_table, int B, int N, int Hkv, int D,
                       int max_blocks, int num_blocks, void *k_cache, void *v_cache,
                       int32_t *ctx_len_out, int32_t *status, tv_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* TV_H_ */
