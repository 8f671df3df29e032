/*
 * treeverify.h -- C ABI of libtreeverify: one-pass verification of a
 * speculative draft tree on an sm_103a GPU (tree structure, depth-indexed
 * RoPE, tree attention over a paged KV cache, tree acceptance).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every function returns an int status: TV_OK (0) or a negative TV_ERR_*
 *   code; tv_last_error() then describes the failure (thread-local string).
 * - "device" pointers are CUDA global memory of the current device; "host"
 *   pointers are ordinary CPU memory.  The caller owns every buffer; the
 *   library allocates no device memory anywhere and keeps no state between
 *   calls apart from per-device property caches.
 * - Device entry points only enqueue work on the caller's stream (a
 *   cudaStream_t passed as void*, NULL = legacy default stream); they never
 *   synchronise and never read device data on the host.  Device-side input
 *   problems (a bad parent array, an out-of-vocabulary token, a negative
 *   prefix length) are not errors of the call: kernels OR TV_DEV_* bits into
 *   the caller's int32 status word (device memory, may be NULL when the
 *   caller does not want it) and skip the offending item, never trapping.
 * - B == 0 is legal everywhere: nothing is launched and TV_OK is returned.
 * - Node 0 of a tree is the root (the last accepted token); N <= 64 nodes,
 *   parent-before-child order (parent[i] < i).
 *
 * Pages cited ("Build the tree attention mask that verifies a draft tree in
 * one pass"; "Implement the lossless speculative sampling verifier for a
 * batch with ragged draft lengths"; "Tree Verification"; "Encode branch
 * histories in masks and positions") are the sources the operations follow.
 */
#ifndef TREEVERIFY_H
#define TREEVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) ------------------------------------ */
#define TV_OK 0
#define TV_ERR_INVALID_ARG (-1)     /* null pointer, bad size or stride     */
#define TV_ERR_MISSING_PARENT (-2)  /* a rank path whose prefix is absent   */
#define TV_ERR_TOO_MANY_NODES (-3)  /* more than max_nodes / 64 tree nodes  */
#define TV_ERR_UNSUPPORTED (-4)     /* shape or dtype this build cannot run */
#define TV_ERR_WORKSPACE (-5)       /* workspace missing or too small       */
#define TV_ERR_CUDA (-6)            /* a CUDA runtime / driver call failed  */

/* ---- device status bits (OR-ed into the caller's int32 status word) ---- */
#define TV_DEV_BAD_TOPOLOGY 1   /* parent[0] != -1 or parent[i] not in [0, i) */
#define TV_DEV_BAD_TOKEN 2      /* draft token outside [0, V): child skipped  */
#define TV_DEV_OUT_OVERFLOW 4   /* walk longer than out_cols: truncated       */
#define TV_DEV_BAD_POSITION 8   /* prefix length < 0 or position >= max_pos   */
#define TV_DEV_TIMEOUT 16       /* a pipeline wait in a kernel exceeded 2 s     */
#define TV_DEV_BAD_BLOCK 32     /* a block-table entry a prefix position uses is outside
                                   [0, num_blocks): those keys and values read as zeros */

/* ---- element types ------------------------------------------------------ */
#define TV_F32 0
#define TV_BF16 1

#define TV_MAX_NODES 64

/* Kernel selection for tv_tree_attn_verify (flags & 3). */
#define TV_ATTN_AUTO 0      /* tensor-core kernel when the shape allows it */
#define TV_ATTN_SIMT 1      /* CUDA-core FP32 kernel (any supported shape)  */
#define TV_ATTN_TCGEN05 2   /* tcgen05/TMEM/TMA kernel; TV_ERR_UNSUPPORTED
                               if the shape or device does not allow it   */
/* Optional flag bit, tcgen05 kernel only: a unit split across CTAs is always
 * merged from the pieces' published partials by the piece that finishes last,
 * never directly from the finishing CTA's accumulator.  Same results up to
 * rounding; for testing the second merge route. */
#define TV_ATTN_PUBLISH_ALL 4
/* Workspace query for tv_tree_attn_verify_rope (Q rotated while it is
 * loaded; the tensor-core kernel then needs Hq/Hkv in {4, 8, 16}).  Not a
 * flag of tv_tree_attn_verify itself. */
#define TV_ATTN_ROPE_Q 8
/* Flag bit, tcgen05 kernel only: units of 129-256 rows (G * N) run on CTA
 * pairs (tcgen05.mma.cta_group::2, each SM loading half of every K/V tile)
 * instead of one SM per unit.  Same results up to rounding; slower than the
 * one-SM kernel on the shapes measured so far. */
#define TV_ATTN_CTA_PAIRS 16
/* Flag bit, tcgen05 kernels: the workspace's arrival counters are already
 * zero, so the call does not clear them first (one memset fewer per call;
 * about 4 us of a 0.28 ms step measured).  Every call that completes leaves
 * them zero again (the piece that merges a split row resets its counter), so
 * the flag holds on a workspace that was zeroed once when allocated and has
 * since been used only by completed calls.  After a call that reported
 * TV_DEV_TIMEOUT, or when the memory held anything else, zero the workspace
 * again (or call without the flag).  Ignored by the CUDA-core kernel and by
 * tv_tree_attn_verify_static, which always clears its counters. */
#define TV_ATTN_WORKSPACE_ZEROED 32

/* Kernel selection of tv_tree_accept_sample and tv_chain_accept_sample. */
#define TV_SAMPLE_AUTO 0        /* TV_SAMPLE_CLUSTER when every request's cluster is resident at
                                   once; else TV_SAMPLE_GRID when a workspace is given and
                                   V <= 1,048,576; else TV_SAMPLE_STREAM with the largest cluster
                                   size that keeps them all resident, else TV_SAMPLE_SINGLE_CTA  */
#define TV_SAMPLE_CLUSTER 1     /* one 8-CTA cluster per request, level weights in shared memory;
                                   TV_ERR_UNSUPPORTED when V > 136,512                            */
#define TV_SAMPLE_SINGLE_CTA 2  /* one CTA per request, rows streamed, weights recomputed per pass */
#define TV_SAMPLE_STREAM 3      /* clusters of 1-8 CTAs per request streaming their row slices, only
                                   chunk totals kept; TV_ERR_UNSUPPORTED when V > 1,048,576         */
#define TV_SAMPLE_GRID 4        /* three kernels over a workspace: a warp per request walks to its
                                   first rejection or leaf, the stop rows' pass runs as uniform
                                   4096-entry items over the whole GPU, a CTA per request draws;
                                   a request whose rejected child has a later valid sibling is
                                   walked again by the TV_SAMPLE_AUTO kernel (the others return at
                                   once).  TV_ERR_INVALID_ARG without a large enough workspace,
                                   TV_ERR_UNSUPPORTED when V > 1,048,576                         */

/* Description of the last failure on this thread ("" if none). */
const char* tv_last_error(void);

/* Library ABI version (major * 100 + minor). */
int tv_version(void);

/*
 * tv_tree_build -- host, synchronous.
 * "Build the tree attention mask ...", sections "The tree." and "The mask.":
 * candidates are rank paths ((0,) = top guess, (0,1) = second guess after
 * the top guess); duplicates are removed; paths are ordered by length, then
 * lexicographically; candidate k of that order becomes node k + 1 (node 0 is
 * the root); parent = node of the path without its last rank; depth = path
 * length; a path whose prefix is not a candidate is rejected; a node attends
 * to itself and its ancestors.
 *
 * ranks     host int32 [offsets[n_paths]]: all paths' ranks concatenated.
 * offsets   host int32 [n_paths + 1]: path k is ranks[offsets[k] .. offsets[k+1]);
 *           an empty path denotes the root and is ignored.
 * max_nodes capacity of the outputs (1..64).
 * parent    host int32 [max_nodes] out: parent[0] = -1.
 * depth     host int32 [max_nodes] out.
 * mask      host uint64 [max_nodes] out: bit j of mask[i] <=> j is i or an
 *           ancestor of i.
 * path_to_node host int32 [n_paths] out (may be NULL): node of each input path.
 * n_nodes   host int32 out: N = 1 + number of distinct non-empty paths.
 * Errors: TV_ERR_INVALID_ARG (null / negative rank / bad offsets),
 * TV_ERR_MISSING_PARENT, TV_ERR_TOO_MANY_NODES.  Zero paths give N = 1.
 */
int tv_tree_build(const int32_t* ranks, const int32_t* offsets, int32_t n_paths,
                  int32_t max_nodes, int32_t* parent, int32_t* depth,
                  uint64_t* mask, int32_t* path_to_node, int32_t* n_nodes);

/*
 * tv_tree_mask -- device, asynchronous.  Batched ancestor rows and positions.
 * "Build the tree attention mask ...", "The mask." (position = prefix length
 * + depth, siblings share a position) and "Tree Verification", "Tree
 * Attention" (parent-before-child flattening).
 *
 * parent    device int32 [B, N] with row stride parent_bstride elements
 *           (0 = one tree shared by all requests).
 * seq_lens  device int32 [B]: prefix length L_b (tokens already cached).
 * n_nodes   device int32 [B] (nullable = N): ragged trees in a bucket of N
 *           ("What interviewers probe next": graph capture needs a fixed
 *           tree shape per batch bucket).  Request b holds nodes
 *           0 .. n_b - 1 (n_b clamped to [1, N]); nodes i >= n_b are absent:
 *           mask 0, depth 0, pos -1, parent[b, i] not read.
 * mask      device uint64 [B, N] out; depth, pos device int32 [B, N] out
 *           (pos = L_b + depth).  A request whose parent row (its first n_b
 *           entries) is not a parent-before-child tree gets zero rows and
 *           TV_DEV_BAD_TOPOLOGY.
 * status    device int32 (nullable), see TV_DEV_*.
 */
int tv_tree_mask(const int32_t* parent, int64_t parent_bstride, const int32_t* seq_lens,
                 const int32_t* n_nodes, int32_t B, int32_t N, uint64_t* mask, int32_t* depth,
                 int32_t* pos, int32_t* status, void* stream);

/*
 * tv_tree_prepare -- device, asynchronous.  tv_tree_mask and RoPE in one
 * launch: the same mask, depth and pos as tv_tree_mask, and the queries
 * and/or tree keys rotated in place at pos exactly as tv_rope_apply would
 * (same bits).  With q = NULL only the tree keys are rotated (the step then
 * uses tv_tree_attn_verify_rope, which rotates Q as it loads it); with both,
 * it replaces tv_tree_mask + tv_rope_apply.
 *
 * parent, parent_bstride, seq_lens, n_nodes, mask, depth, pos: as in
 *           tv_tree_mask.
 * q         device [B, N, Hq, head_dim] (dtype), rotated in place (nullable).
 * k_tree    device [B, N, Hkv, head_dim] (dtype), rotated in place
 *           (nullable; both NULL: only the mask part).  head_dim in
 *           {16, 32, 64, 128, 256}.
 * cos_sin   device float32 [max_pos, 2, head_dim/2] from tv_rope_table.
 * A position outside [0, max_pos) other than -1 leaves the row untouched and
 * sets TV_DEV_BAD_POSITION; -1 (absent node) leaves it silently.
 */
int tv_tree_prepare(const int32_t* parent, int64_t parent_bstride, const int32_t* seq_lens,
                    const int32_t* n_nodes, int32_t B, int32_t N, uint64_t* mask, int32_t* depth,
                    int32_t* pos, void* q, int32_t Hq, void* k_tree, int32_t Hkv, int32_t head_dim,
                    int32_t dtype, const float* cos_sin, int32_t max_pos, int32_t* status, void* stream);

/*
 * tv_rope_table -- device, asynchronous.  Fills the rotary table used by
 * tv_rope_apply: cos_sin float32 [max_pos, 2, D/2]; row p holds
 * cos(p * base^(-2k/D)) for k < D/2 followed by the matching sines, each
 * evaluated in float64 and rounded once to float32.
 */
int tv_rope_table(float* cos_sin, int32_t max_pos, int32_t head_dim, double base, void* stream);

/*
 * tv_rope_apply -- device, asynchronous, in place.
 * "Build the tree attention mask ...", "What interviewers probe next" and
 * "Common mistakes" (RoPE must rotate a node at its depth, not at its
 * flattened index); "Encode branch histories ..." (positional features
 * follow the model's position semantics).  Rotate-half convention: for each
 * row x of length D, (x1, x2) = (x[:D/2], x[D/2:]) becomes
 * (x1 cos - x2 sin, x2 cos + x1 sin) at position pos[b, i], math in float32.
 *
 * q       device [B, N, Hq, D] (dtype), rotated in place.
 * k_tree  device [B, N, Hkv, D] (dtype), rotated in place (may be NULL).
 * pos     device int32 [B, N] (from tv_tree_mask).
 * cos_sin device float32 [max_pos, 2, D/2] from tv_rope_table.
 * A position outside [0, max_pos) leaves the row untouched and sets
 * TV_DEV_BAD_POSITION, except -1 (an absent node of a ragged tree), which
 * leaves it untouched silently.  D in {16, 32, 64, 128, 256}; B*N*(Hq+Hkv)*D/16 < 2^31
 * (else TV_ERR_UNSUPPORTED).
 */
int tv_rope_apply(void* q, void* k_tree, const int32_t* pos, const float* cos_sin,
                  int32_t max_pos, int32_t B, int32_t N, int32_t Hq, int32_t Hkv,
                  int32_t head_dim, int32_t dtype, int32_t* status, void* stream);

/*
 * tv_tree_attn_workspace_size -- host.  Bytes of device workspace that
 * tv_tree_attn_verify needs for this shape, kernel choice (flags) and grid
 * (num_ctas, 0 = one wave of the current device).  Does not depend on the
 * prefix lengths.
 */
int tv_tree_attn_workspace_size(int32_t B, int32_t N, int32_t Hq, int32_t Hkv,
                                int32_t head_dim, int32_t dtype, int32_t block_size,
                                int32_t num_ctas, int32_t flags, size_t* bytes);

/*
 * tv_tree_attn_verify -- device, asynchronous.  One-pass tree attention.
 * "Tree Verification", "Tree Attention": every node attends to the whole
 * cached prefix, to its root-path ancestors and to itself, nothing else;
 * "Build the tree attention mask ...", "The mask.": the step mask is
 * [prefix all true | tree mask] and a kernel may take the tree part as
 * per-node ancestor rows.  Output row (b, i, h) is
 *   softmax(scale * q . K^T) V  over keys = prefix 0..L_b-1 of request b
 *   (KV head h / (Hq/Hkv)) followed by the tree nodes j with bit j of
 *   mask[b, i] set.  A row whose key set is empty (L_b = 0 and a zero mask
 *   row, i.e. an absent node) is written as zeros with lse = -inf; an absent
 *   node with L_b > 0 attends to the prefix only.
 * q and k_tree must already be rotated (tv_rope_apply); the cached prefix
 * keys are stored rotated.
 *
 * q          device [B, N, Hq, D] (dtype).
 * k_cache,   device [num_blocks, Hkv, block_size, D] (dtype): position t of
 * v_cache    request b is block block_table[b, t / block_size], slot
 *            t % block_size.  Slots >= L_b of a used block must hold finite
 *            values (they are read and weighted by exactly zero).
 * block_table device int32 [B, max_blocks]; entries >= ceil(L_b/block_size)
 *            are never read; an entry that is read but lies outside
 *            [0, num_blocks) reads as zero keys and values and sets
 *            TV_DEV_BAD_BLOCK.
 * seq_lens   device int32 [B], 0 <= L_b <= max_blocks * block_size.
 * k_tree,    device [B, N, Hkv, D] (dtype): node K/V (node 0 = root).
 * v_tree
 * mask       device uint64 [B, N] with row stride mask_bstride elements
 *            (0 = shared); bit j of mask[b, i] <=> node i may see node j.
 * scale      softmax scale (e.g. 1/sqrt(D)).
 * out        device [B, N, Hq, D] (dtype) out; 32-byte aligned (and q
 *            16-byte aligned) on the tensor-core path, else
 *            TV_ERR_INVALID_ARG.
 * lse        device float32 [B, N, Hq] out (nullable): natural-log softmax
 *            normaliser of each row.
 * workspace  device buffer of at least tv_tree_attn_workspace_size bytes,
 *            256-byte aligned; its contents on entry are irrelevant (the
 *            tensor-core path clears its arrival counters in it with a
 *            cudaMemsetAsync on `stream`), except with
 *            TV_ATTN_WORKSPACE_ZEROED, which asks for zero counters and
 *            skips the clearing.
 * flags      TV_ATTN_* kernel selection, optionally | TV_ATTN_PUBLISH_ALL
 *            | TV_ATTN_CTA_PAIRS | TV_ATTN_WORKSPACE_ZEROED.
 * num_ctas   persistent grid size (0 = one wave of the current device);
 *            must equal the value given to tv_tree_attn_workspace_size.
 * status     device int32 (nullable): TV_DEV_TIMEOUT if a pipeline wait of
 *            the tensor-core kernel gave up (the output is then incomplete).
 * Supported: N <= 64, D in {64, 128, 256}, dtype TV_F32 or TV_BF16,
 * Hq % Hkv == 0.  The tensor-core kernel needs an sm_10x device, bf16,
 * D = 128, G = Hq/Hkv dividing 128, G * N <= 512, block_size a multiple of 16
 * that divides 64 or is a multiple of 64, and num_blocks * Hkv * block_size
 * < 2^31; TV_ATTN_AUTO falls back to the CUDA-core kernel otherwise.
 * TV_ERR_UNSUPPORTED as well when the work plan could reach 2^31 tiles:
 * units x (ceil(max_blocks * block_size / 64) + 1 + c), where units =
 * B * Hkv * ceil(G * N / rows per unit) and c is the per-unit cost in tiles
 * (at most 6 for the tensor-core kernel, 0 for the CUDA-core one).
 */
int tv_tree_attn_verify(const void* q, const void* k_cache, const void* v_cache,
                        int64_t num_blocks, int32_t block_size,
                        const int32_t* block_table, int32_t max_blocks,
                        const int32_t* seq_lens, const void* k_tree, const void* v_tree,
                        const uint64_t* mask, int64_t mask_bstride,
                        int32_t B, int32_t N, int32_t Hq, int32_t Hkv, int32_t head_dim,
                        int32_t dtype, float scale, void* out, float* lse,
                        void* workspace, size_t workspace_bytes, int32_t num_ctas,
                        int32_t flags, int32_t* status, void* stream);

/*
 * tv_tree_attn_verify_rope -- device, asynchronous.  tv_tree_attn_verify with
 * RoPE of the queries fused into the kernels' Q load ("Build the tree
 * attention mask ...", "What interviewers probe next": a node is rotated at
 * its depth position; the separate rope step is one read and write of Q the
 * fused load saves).  q is given unrotated and is not modified; each row is
 * rotated at L_b + depth, depth = popcount(mask row) - 1, with the table
 * cos_sin [max_pos, 2, head_dim/2] and exactly the arithmetic and rounding of
 * tv_rope_apply, so the outputs have the same bits as tv_rope_apply followed
 * by tv_tree_attn_verify.  k_tree must already be rotated (tv_tree_prepare,
 * or tv_rope_apply with q = NULL).  A zero mask row (absent node) is not
 * rotated; a position >= max_pos leaves the row unrotated and sets
 * TV_DEV_BAD_POSITION.  Workspace: tv_tree_attn_workspace_size with flags |
 * TV_ATTN_ROPE_Q (the tensor-core kernel takes Hq/Hkv in {4, 8, 16} here; the
 * CUDA-core kernel any).  Other arguments as in tv_tree_attn_verify.
 */
int tv_tree_attn_verify_rope(const void* q, const void* k_cache, const void* v_cache,
                             int64_t num_blocks, int32_t block_size,
                             const int32_t* block_table, int32_t max_blocks,
                             const int32_t* seq_lens, const void* k_tree, const void* v_tree,
                             const uint64_t* mask, int64_t mask_bstride,
                             const float* cos_sin, int32_t max_pos,
                             int32_t B, int32_t N, int32_t Hq, int32_t Hkv, int32_t head_dim,
                             int32_t dtype, float scale, void* out, float* lse,
                             void* workspace, size_t workspace_bytes, int32_t num_ctas,
                             int32_t flags, int32_t* status, void* stream);

/*
 * tv_tree_attn_verify_static -- device, asynchronous; allocation-free variant
 * of tv_tree_attn_verify.  No page describes it: it exists for callers that
 * cannot provide device memory when they verify a tree -- a serving loop that
 * reserves all memory at start-up and forbids allocation afterwards, a host
 * runtime without a device allocator, or code that must not call cudaMalloc
 * because it can synchronise the device.  Same arguments and results as
 * tv_tree_attn_verify without the workspace: the scratch (tile plan and
 * split partials) is a fixed array of tv_tree_attn_static_workspace_bytes()
 * (32 MiB) that the library places in device memory of every GPU that loads
 * it, held until the process exits.
 *
 * num_ctas   0 = the widest grid, at most one wave, whose scratch fits the
 *            array; an explicit grid whose scratch exceeds the array, or a
 *            shape whose plan alone does not fit, returns TV_ERR_WORKSPACE.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  After a cudaDeviceReset the next call looks the address up again
 * (the device's context has changed), so make that call outside a capture
 * too.  The call allocates nothing (no cudaMalloc / cudaFree).  Every call
 * uses the same array, so calls that can overlap on the GPU (different
 * streams, or graphs replayed concurrently) race and must be serialised by the
 * caller; the array needs no clearing between calls (everything read is
 * written earlier in the same call).
 */
int tv_tree_attn_verify_static(const void* q, const void* k_cache, const void* v_cache,
                               int64_t num_blocks, int32_t block_size,
                               const int32_t* block_table, int32_t max_blocks,
                               const int32_t* seq_lens, const void* k_tree, const void* v_tree,
                               const uint64_t* mask, int64_t mask_bstride,
                               int32_t B, int32_t N, int32_t Hq, int32_t Hkv, int32_t head_dim,
                               int32_t dtype, float scale, void* out, float* lse,
                               int32_t num_ctas, int32_t flags, int32_t* status, void* stream);

/* Size in bytes of the fixed scratch array used by tv_tree_attn_verify_static
 * (no page describes it; see above). */
size_t tv_tree_attn_static_workspace_bytes(void);

/*
 * tv_tree_accept_greedy -- device, asynchronous.
 * "Build the tree attention mask ...", "The mask." (walk from the root while
 * some child's draft token equals the target's choice after the current
 * node; every visited node emits the target's choice) and "Encode branch
 * histories ..." (node i's logits predict its children).  Children are tried
 * in ascending node index; the target's choice is the largest logit, ties to
 * the lowest vocabulary index.
 *
 * logits        device float32 [B, N, V] (row stride V) or NULL; then
 * target_argmax device int32 [B, N] gives the choices directly.
 * tokens        device int32 [B, N]: draft token of node i (column 0 unused).
 * parent        device int32 [B, N], row stride parent_bstride (0 = shared).
 * n_nodes       device int32 [B] (nullable = N): nodes >= n_nodes[b] absent.
 * out           device int32 [B, out_cols] out: emitted tokens, -1 padded.
 * n_out         device int32 [B] out: accepted drafts + 1.
 * path          device int32 [B, out_cols] out (nullable): node at which
 *               each token was emitted (root first), -1 padded.
 * status        device int32 (nullable), TV_DEV_OUT_OVERFLOW if a walk does
 *               not fit in out_cols (out_cols >= max depth + 1 avoids it).
 */
int tv_tree_accept_greedy(const float* logits, const int32_t* target_argmax,
                          const int32_t* tokens, const int32_t* parent,
                          int64_t parent_bstride, const int32_t* n_nodes,
                          int32_t B, int32_t N, int32_t V, int32_t* out,
                          int32_t* n_out, int32_t* path, int32_t out_cols,
                          int32_t* status, void* stream);

/*
 * tv_tree_accept_sample -- device, asynchronous.  Lossless stochastic walk.
 * "Implement the lossless speculative sampling verifier ...", "A strong
 * answer" (accept x iff u * q(x) < p(x), no division; first rejection stops
 * the chain; replacement from the normalised residual max(0, p - q); bonus
 * from p after the last accepted node; p = q guard) and "What interviewers
 * probe next" (on a tree: after a rejection the target at that node becomes
 * the normalised residual and the next sibling is tested against it);
 * "Tree Verification", "Accepting on a Tree" (top-down walk, a leaf earns the
 * bonus).
 *
 * Exact arithmetic (both this kernel and any checker follow it bit for bit):
 *  - level 0 at a node: accept child x iff (double)u * (double)q(x) < (double)p(x);
 *  - integer images P = rint(p * 2^40), Q = rint(q * 2^40) (half to even);
 *    after a rejection at level m (scale S_0 = 2^40, S_m = W_m for m >= 1):
 *    w_{m+1} = max(0, w_m - floor((S_m * Q + 2^39) / 2^40)), w_0 = P,
 *    W_{m+1} = sum w_{m+1}; if W_{m+1} == 0 the level is not advanced;
 *  - level m >= 1: accept iff fl64(fl64(u * q(x)) * W_m) < w_m(x);
 *  - the final draw (replacement, or bonus from p at level 0 with W = sum P)
 *    returns min(#{x : prefix_sum_w(x) < ceil(fl64(u_final * W))}, V - 1).
 * Contract: every p and q row sums to at most 2 and holds no negative entry
 * (probability rows; an entry below zero is taken as 0).
 *
 * p, q      device float32 [B, N, V]: target distribution after node i and the
 *           draft distribution node i's children were drawn from.
 * tokens    device int32 [B, N]; parent as in greedy; n_nodes [B] (nullable).
 * u_accept  device float32 [B, N]: uniform used when node i is tested.
 * u_final   device float32 [B]: uniform of the replacement / bonus draw.
 * out, n_out, path, out_cols, status: as in tv_tree_accept_greedy.  Tokens
 * outside [0, V) are skipped and flagged TV_DEV_BAD_TOKEN.
 * flags     TV_SAMPLE_*: every kernel gives bit-identical results.  The
 *           cluster kernel splits each row over 8 CTAs and keeps the current
 *           level's weights and q in shared memory (12 bytes per vocabulary
 *           entry), so repeated rejections at a node cost one shared-memory
 *           pass each.  The streaming clusters re-read their slice from
 *           memory at every pass and keep only 256-element chunk totals, so
 *           large batches stay resident.  The grid sampler spreads the stop
 *           rows' pass evenly over the GPU (a request that rejected reads
 *           two rows, one that reached a leaf one).  Unknown flags give
 *           TV_ERR_INVALID_ARG.
 * workspace device scratch (nullable), 16-byte aligned, of workspace_bytes
 *           >= tv_accept_sample_workspace_size(B, N, V) for the grid
 *           sampler; its contents need no initialisation and are not read
 *           after the call.  NULL (or a smaller size) keeps TV_SAMPLE_AUTO
 *           to the single-launch kernels.  Calls that overlap on the GPU
 *           need their own workspaces.
 */
int tv_tree_accept_sample(const float* p, const float* q, const int32_t* tokens,
                          const int32_t* parent, int64_t parent_bstride,
                          const int32_t* n_nodes, const float* u_accept,
                          const float* u_final, int32_t B, int32_t N, int32_t V,
                          int32_t* out, int32_t* n_out, int32_t* path, int32_t out_cols,
                          int32_t flags, void* workspace, size_t workspace_bytes,
                          int32_t* status, void* stream);

/*
 * tv_accept_sample_workspace_size -- host.  Bytes of the grid sampler's
 * workspace for B requests of N nodes over V vocabulary entries: 16 per
 * request, and 16 per request and 4096-entry chunk of a row; 0 when B <= 0
 * or V <= 0.
 */
size_t tv_accept_sample_workspace_size(int32_t B, int32_t N, int32_t V);

/*
 * tv_accept_sample_uses_grid -- host (queries the current device).  Sets
 * *grid to 1 when a sampler call with these sizes, flags and a workspace of
 * workspace_bytes (0: none) takes the grid sampler (its three kernels plus a
 * walk of the requests they leave), else 0.  TV_ERR_INVALID_ARG for unknown
 * flags or bad sizes.
 */
int tv_accept_sample_uses_grid(int32_t B, int32_t N, int32_t V, int32_t flags,
                               size_t workspace_bytes, int32_t* grid);

/*
 * tv_chain_accept_sample -- device, asynchronous.  The verifier page's own
 * call shape, "Implement the lossless speculative sampling verifier ...",
 * "A strong answer" (verify(draft, q, p, num_draft, u, u_final): ragged draft
 * chains, first rejection stops the chain, replacement from the residual,
 * bonus after a fully accepted chain).  The same walk, arithmetic and kernels
 * as tv_tree_accept_sample on the chain whose node j + 1 is draft j (node 0
 * the last accepted token), bit for bit; the arrays are read where they are
 * (nothing is copied or allocated).
 *
 * p         device float32 [B, K + 1, V]: the target after each prefix (row K:
 *           after the whole chain, the bonus row).
 * q         device float32 [B, K, V]: draft j was drawn from q[b, j].
 * draft     device int32 [B, K]; num_draft device int32 [B] (nullable = K;
 *           clamped to [0, K]): request b's drafts are draft[b, 0 .. num_draft).
 * u         device float32 [B, K]: uniform of the test of draft j.
 * u_final   device float32 [B]: uniform of the replacement / bonus draw.
 * out       device int32 [B, out_cols] out: emitted tokens, -1 padded;
 * n_out     device int32 [B] out: accepted drafts + 1.
 * K in [0, TV_MAX_NODES - 1]; flags, workspace (size for N = K + 1) and
 * status as in tv_tree_accept_sample.
 */
int tv_chain_accept_sample(const float* p, const float* q, const int32_t* draft,
                           const int32_t* num_draft, const float* u, const float* u_final,
                           int32_t B, int32_t K, int32_t V, int32_t* out, int32_t* n_out,
                           int32_t out_cols, int32_t flags, void* workspace,
                           size_t workspace_bytes, int32_t* status, void* stream);

/*
 * tv_kv_commit -- device, asynchronous.  Copies the accepted path's tree K/V
 * into the paged cache.  "Build the tree attention mask ...", "What it
 * costs." (tree K/V in scratch, the accepted path copied into the cache);
 * "Tree Verification", "The Cost Side".  Node path[b, j] (j < n_out[b]) sits
 * at depth j: its K and V rows, every KV head, go to cache position
 * L_b + j, i.e. block block_table[b, (L_b + j) / block_size], slot
 * (L_b + j) % block_size.  The tree keys are copied as given (after
 * tv_rope_apply they are rotated at L_b + depth, their cache position).
 *
 * k_cache, v_cache  device [num_blocks, Hkv, block_size, D] (dtype), written.
 * block_table       device int32 [B, max_blocks]; the caller has placed
 *                   blocks for positions up to L_b + n_out[b] - 1.
 * seq_lens          device int32 [B]: L_b (read).
 * new_seq_lens      device int32 [B] out (nullable, must not alias
 *                   seq_lens): L_b + n_out[b], or L_b + j when step j is the
 *                   first that cannot be committed (below).
 * k_tree, v_tree    device [B, N, Hkv, D] (dtype).
 * path              device int32 [B, path_cols]: the accepted path as
 *                   tv_tree_accept_* return it (node indices, root first).
 * n_out             device int32 [B]: path length per request (values are
 *                   clamped to [0, path_cols]).
 * The first path step whose node index is outside [0, N) (TV_DEV_BAD_TOPOLOGY)
 * or whose position is beyond the block table or maps to a table entry
 * outside [0, num_blocks) (TV_DEV_OUT_OVERFLOW) ends the commit: the steps
 * before it are copied, nothing from it on, and new_seq_lens counts only
 * the copied steps, so the next step never treats unwritten slots as
 * prefix.  D * element
 * size must be a multiple of 16 bytes and the K/V buffers 16-byte aligned.
 * No page defines a separate entry point: it is the copy the mask page's
 * serving loop performs after acceptance.
 */
int tv_kv_commit(void* k_cache, void* v_cache, int64_t num_blocks, int32_t block_size,
                 const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                 int32_t* new_seq_lens, const void* k_tree, const void* v_tree,
                 const int32_t* path, int32_t path_cols, const int32_t* n_out, int32_t B,
                 int32_t N, int32_t Hkv, int32_t head_dim, int32_t dtype, int32_t* status,
                 void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TREEVERIFY_H */
