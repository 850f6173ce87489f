/*
 * spec_verify.h -- C ABI of libspecverify.so, the target-side verification
 * step of speculative decoding on one GPU (sm_103a).
 *
 * The step has two parts, both defined by the pages this library follows:
 *
 *   spec_verify_attn    one multi-row attention pass over the proposed block
 *                       ("Drafters and Speculative Decoding: Useful Tokens,
 *                       Correct State", section "From a proposed block to a
 *                       causal target pass"), with a draft-tree visibility
 *                       mask ("Speculative Decoding" (atlas), section
 *                       "Chains, trees and visibility"), computed as split-K
 *                       flash-decoding partials plus a log-sum-exp combine
 *                       ("Speculative Token Decoupling: Asynchronous
 *                       Verification via Flash-Decoding", section 03).
 *   spec_accept_sample  the lossless acceptance sampler: target distribution
 *                       p with temperature / top-k / top-p, left-to-right
 *                       test u*q(x) < p(x) on shifted rows, residual
 *                       norm(max(0, p - q)) at the first rejection, bonus
 *                       token when every draft survives, greedy mode
 *                       ("Speculative Decoding" (atlas), sections "One round
 *                       and shifted logits", "Exact sampling: account for
 *                       every probability", "Greedy, sampling and the real
 *                       sampler"; "Drafters and Speculative Decoding",
 *                       section "Sampling needs a correction rule").
 *
 * Conventions for every call:
 *   - Array arguments are DEVICE pointers owned by the caller, in the layout
 *     given beside each argument (row-major, innermost last).  The library
 *     keeps no pointer after a call returns.
 *   - The library allocates no memory.  Scratch comes from a caller-provided
 *     workspace whose size a *_workspace_size() call returns.  Workspaces
 *     hold self-resetting counters: zero-fill a workspace once when you
 *     allocate it; every completed call leaves it ready for the next one.
 *     Concurrent calls must not share a workspace.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  No call synchronises.  Calls may be captured in CUDA graphs.
 *   - Argument and shape errors are detected on the host before any launch
 *     and return SPEC_EINVAL; shapes outside the supported envelope return
 *     SPEC_EUNSUPPORTED; a failed launch returns SPEC_ECUDA.  Data-dependent
 *     conditions are reported per sequence in status_per_seq (bits below).
 *   - Device-side waits are bounded; a wait that runs out sets the error
 *     word that spec_workspace_error() reads, and the call's outputs are then
 *     unspecified.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_EINVAL = 1,        /* bad pointer, size or parameter */
  SPEC_EUNSUPPORTED = 2,  /* valid request outside what the kernels implement */
  SPEC_ECUDA = 3,         /* a CUDA runtime/driver call failed */
  SPEC_ETIMEOUT = 4       /* a bounded device-side wait ran out (error word) */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* status_per_seq bits (OR-ed). */
#define SPEC_SEQ_QZERO 1       /* a proposed token had q(x) == 0; it was accepted iff p(x) > 0 */
#define SPEC_SEQ_NONFINITE 2   /* a target logit was NaN or +inf; that sequence's outputs are -1 */
#define SPEC_SEQ_RESID_ZERO 4  /* residual mass was 0 after a rejection; the draw used p */
#define SPEC_SEQ_BAD_TREE 8    /* parent array is not a tree in storage order */

/* Error words written to a workspace by a bounded wait that ran out. */
#define SPEC_ERR_MBAR_TIMEOUT 0x100

/* Human-readable name of a status code (static string). */
const char* spec_status_str(spec_status s);

/* ------------------------------------------------------------------------
 * spec_tree_prepare -- visibility of a flattened draft tree.
 * "Speculative Decoding" (atlas), "Chains, trees and visibility": each node
 * sees the accepted prefix, its ancestors and itself; position ids follow
 * depth; a parent array plus an ancestor mask state this.
 *
 *   parent   [B,R] int32, node 0 is the root/pending anchor (parent -1), every
 *            other node i has 0 <= parent[i] < i.  NULL means a chain
 *            (parent[i] = i - 1), the causal case.
 *   ctx_len  [B] int32, committed tokens before the block (>= 0).
 *   anc_mask [B,R] uint64 out: bit j set iff node j is node i or an ancestor.
 *   pos_ids  [B,R] int32 out (nullable): ctx_len[b] + depth(i).
 *   status_per_seq [B] int32 out (nullable): SPEC_SEQ_BAD_TREE if the parent
 *            row breaks the rule above (mask/pos of that row are then 0).
 *   1 <= R <= 64.
 * ---------------------------------------------------------------------- */
spec_status spec_tree_prepare(const int32_t* parent, const int32_t* ctx_len, int B, int R,
                              uint64_t* anc_mask, int32_t* pos_ids, int32_t* status_per_seq,
                              void* stream);

/* ------------------------------------------------------------------------
 * spec_verify_attn -- multi-row, tree-masked, paged GQA attention as split-K
 * flash-decoding partials plus a log-sum-exp combine.
 *
 *   q          [B,R,Hq,D]   dtype (bf16, or fp32 for the CUDA-core path)
 *   k_cache,
 *   v_cache    [num_pages,page_size,Hkv,D] dtype; the R block rows of
 *              sequence b are already stored at positions ctx_len[b] ..
 *              ctx_len[b]+R-1 of its page list.
 *   block_table[B,max_pages] int32: page ids of sequence b in order.  Entries
 *              past the sequence's last page are not read.
 *   ctx_len    [B] int32: committed positions, all visible to every row.
 *   anc_mask   [B,R] uint64: block position ctx+j is visible to row i iff bit
 *              j of anc_mask[b,i] is set (spec_tree_prepare's output).  NULL
 *              means a chain: row i sees block rows 0 .. i (the causal block,
 *              no spec_tree_prepare launch needed).
 *   scale      softmax scale; <= 0 selects 1/sqrt(D).
 *   num_splits KV chunks per (sequence, KV head); 0 lets the library choose.
 *   workspace  >= spec_verify_attn_workspace_size(...) bytes, 256-B aligned.
 *   out        [B,R,Hq,D] dtype.
 *   lse_out    [B,R,Hq] fp32 natural-log LSE of the scaled scores (nullable).
 *
 * Query head h reads KV head h / (Hq/Hkv).  Supported: D in {64,128};
 * bf16 needs D == 128, page_size % 16 == 0, 16-byte aligned cache rows;
 * fp32 any page_size; R*Hq/Hkv <= 512; R <= 64; B <= 65535.
 * ---------------------------------------------------------------------- */
size_t spec_verify_attn_workspace_size(int B, int R, int Hq, int Hkv, int D, int page_size,
                                       int max_pages, int num_splits);

/* The split count the library would use (resolves num_splits == 0). */
int spec_verify_attn_num_splits(int B, int R, int Hq, int Hkv, int D, int page_size,
                                int max_pages, int num_splits);

spec_status spec_verify_attn(const void* q, const void* k_cache, const void* v_cache,
                             spec_dtype dtype, int page_size, int num_pages,
                             const int32_t* block_table, int max_pages,
                             const int32_t* ctx_len, const uint64_t* anc_mask,
                             int B, int R, int Hq, int Hkv, int D, float scale, int num_splits,
                             void* workspace, size_t workspace_bytes,
                             void* out, float* lse_out, void* stream);

/* The two phases of spec_verify_attn as separate calls, with the same
 * arguments: spec_verify_attn_partials launches the split-K pass (one partial
 * output and log-sum-exp per KV chunk, kept in `workspace`); a following
 * spec_verify_attn_combine on the same stream, with the same shapes and
 * workspace, merges them into `out` / `lse_out` ("Speculative Token
 * Decoupling: Asynchronous Verification via Flash-Decoding", section 03:
 * split-K attention).  The combine reads only ctx_len and the workspace;
 * q, k_cache, v_cache, block_table and anc_mask may be NULL there. */
spec_status spec_verify_attn_partials(const void* q, const void* k_cache, const void* v_cache,
                                      spec_dtype dtype, int page_size, int num_pages,
                                      const int32_t* block_table, int max_pages,
                                      const int32_t* ctx_len, const uint64_t* anc_mask,
                                      int B, int R, int Hq, int Hkv, int D, float scale,
                                      int num_splits, void* workspace, size_t workspace_bytes,
                                      void* stream);

spec_status spec_verify_attn_combine(const void* q, const void* k_cache, const void* v_cache,
                                     spec_dtype dtype, int page_size, int num_pages,
                                     const int32_t* block_table, int max_pages,
                                     const int32_t* ctx_len, const uint64_t* anc_mask,
                                     int B, int R, int Hq, int Hkv, int D, float scale,
                                     int num_splits, void* workspace, size_t workspace_bytes,
                                     void* out, float* lse_out, void* stream);

/* ------------------------------------------------------------------------
 * spec_debug_attn_fault -- TEST ONLY: make the bounded device waits of the
 * attention partial passes run out on purpose.  The pages have no
 * counterpart; this exists so that a test can show that a wait that runs out
 * ends the kernel with an error word instead of hanging the GPU.
 *
 *   withhold_stage  >= 0: in every partial-pass CTA launched from now on, the
 *                   copy warps never signal that K/V stage withhold_stage has
 *                   landed, so the waits on it (and those behind it) run out;
 *                   -1: normal operation.
 *   wait_limit_ns   bound of every wait of the partial passes; 0 restores the
 *                   default (2 s).
 * The setting is process-wide and applies to every later call on every
 * device; restore it with (-1, 0).  A CTA whose wait ran out sets
 * SPEC_ERR_MBAR_TIMEOUT in the workspace error word (spec_workspace_error),
 * lets its own copies and tensor-core operations finish, frees its tensor
 * memory and returns; the call's outputs are then unspecified.
 * ---------------------------------------------------------------------- */
spec_status spec_debug_attn_fault(int withhold_stage, unsigned long long wait_limit_ns);

/* ------------------------------------------------------------------------
 * spec_verify_attn_noalloc -- spec_verify_attn for callers that cannot
 * allocate device memory.  (The pages have no counterpart: this is a
 * deployment convenience, not part of the method.)
 *
 * Some callers cannot provide a workspace: a host application that passes a
 * plugin nothing but its input and output buffers, a serving loop that may
 * not allocate once it has started (its memory budget is fixed), or code
 * that must not touch an allocator while the GPU is in use by others.  This
 * call takes the same arguments as spec_verify_attn minus the workspace and
 * keeps its split-K scratch in a fixed array of SPEC_NOALLOC_SCRATCH_BYTES
 * compiled into the library.  That array occupies memory on every GPU that
 * loads the library until the process exits.
 *
 *   - It allocates nothing and calls no allocating routine.  The first call on
 *     each device looks up the array's device address (with that device
 *     current) and caches it; make that first call before any stream capture.
 *   - Problems whose scratch (spec_verify_attn_workspace_size) exceeds
 *     SPEC_NOALLOC_SCRATCH_BYTES are refused with SPEC_EUNSUPPORTED before any
 *     launch; use spec_verify_attn with your own workspace for those.
 *   - All calls share the one array and it keeps whatever the last call left
 *     there.  Calls whose GPU work overlaps (different streams, or different
 *     host threads on one device without ordering) race on it and give wrong
 *     results: order them on one stream.
 *   - The cached address belongs to the device's current context: calls must
 *     not span a reset of the device (cudaDeviceReset).
 *   - Outputs equal spec_verify_attn's for the same arguments.  A bounded
 *     device wait that runs out is recorded in an error word at the head of
 *     the fixed array, which each call clears when it starts; read it with
 *     spec_verify_attn_noalloc_error after the call (the outputs of a call
 *     whose word is nonzero are unspecified, as for spec_verify_attn).
 * ---------------------------------------------------------------------- */
#define SPEC_NOALLOC_SCRATCH_BYTES (8u << 20)

spec_status spec_verify_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                     spec_dtype dtype, int page_size, int num_pages,
                                     const int32_t* block_table, int max_pages,
                                     const int32_t* ctx_len, const uint64_t* anc_mask,
                                     int B, int R, int Hq, int Hkv, int D, float scale,
                                     int num_splits, void* out, float* lse_out, void* stream);

/* The error word of the last spec_verify_attn_noalloc call on the current
 * device (0, or SPEC_ERR_MBAR_TIMEOUT), copied to *host_err.  Synchronises
 * `stream`, on which that call was enqueued; allocates nothing. */
spec_status spec_verify_attn_noalloc_error(int32_t* host_err, void* stream);

/* ------------------------------------------------------------------------
 * Sampler settings, as actually served ("Greedy, sampling and the real
 * sampler": p and q must include the served transforms).
 *   temperature > 0 (ignored when greedy);  top_k: 0 or >= V disables, else
 *   the k largest logits stay (ties: lower id first);  top_p in (0,1]: 1
 *   disables, else the shortest (prob desc, id asc) prefix of the top-k
 *   distribution with mass >= top_p stays, crossing token included;
 *   greedy != 0: argmax verification;  eos_id >= 0: emission stops after the
 *   first EOS token (-1 disables).
 * ---------------------------------------------------------------------- */
typedef struct {
  float temperature;
  int32_t top_k;
  float top_p;
  int32_t greedy;
  int32_t eos_id;
} spec_sampler;

/* Workspace of spec_accept_sample / _tree for B sequences of R rows (N
 * nodes) over a vocabulary of V; 0 for invalid sizes.  The per-sequence
 * counters sit at one place for every shape (room for 65536 sequences after
 * the 256-byte error header), so a zero-filled workspace serves any later
 * call whose own size fits in it, whatever its B, R or V.
 *
 * When many rows are sampled at once (B R cluster(V) > 2 x the SM count,
 * cluster(V) = min(8, ceil(V / 16384))) with truncation, each row is handled
 * by one CTA that sweeps it once (maximum, Z and a candidate list of the ids
 * at or above a sampled floor) and works on the list.  A workspace of
 * spec_accept_sample_workspace_size_two_pass(B, R, V) bytes (about 260 KB
 * per row more) selects the two-pass variant instead: a pre-pass sweeps
 * every row from HBM once over all SMs (maximum, Z and the candidate list of
 * each warp range), then one CTA per row finishes it.  The results are the
 * same; the one-kernel variant is the faster one, alone and next to
 * concurrent HBM-bound work, so it is the default. */
size_t spec_accept_sample_workspace_size(int B, int R, int V);
size_t spec_accept_sample_workspace_size_two_pass(int B, int R, int V);

/* ------------------------------------------------------------------------
 * spec_accept_sample -- chain verification of B sequences.
 *
 *   target_logits [B,R,V] fp32, R = gamma + 1: row 0 is scored after the
 *                 pending anchor, row i after draft i; row i checks draft
 *                 i+1 and row gamma gives the bonus (shifted logits).
 *   draft_probs   [B,R-1,V] fp32: row i is the distribution that actually
 *                 proposed draft i+1 (already transformed).  May be NULL in
 *                 greedy mode.
 *   draft_tokens  [B,R-1] int32 in [0,V).
 *   uniforms      [B,R] fp32 in [0,1): u[i] tests draft i+1, u[R-1] is the
 *                 single draw used by the correction or the bonus token.
 *   accepted_len  [B] int32 out: drafts accepted (0..R-1).
 *   emitted       [B,R] int32 out: accepted drafts then the correction or
 *                 bonus token; -1 after the last emitted token.
 *   p_out         [B,R,V] fp32 out (nullable): the target distribution p of
 *                 every row (not written in greedy mode).
 *   status_per_seq[B] int32 out (nullable): SPEC_SEQ_* bits.
 *
 * A token is accepted iff u*q(x) < p(x) (the event u < min(1, p/q)); the
 * correction is the first id t whose ascending running sum of
 * max(0, p - q) exceeds u_final * sum; the bonus draws from p the same way.
 * 1 <= B <= 65536, 1 <= R <= 64, 1 <= V <= 172032.
 * ---------------------------------------------------------------------- */
spec_status spec_accept_sample(const float* target_logits, const float* draft_probs,
                               const int32_t* draft_tokens, const float* uniforms,
                               int B, int R, int V, const spec_sampler* cfg,
                               void* workspace, size_t workspace_bytes,
                               int32_t* accepted_len, int32_t* emitted, float* p_out,
                               int32_t* status_per_seq, void* stream);

/* ------------------------------------------------------------------------
 * spec_accept_sample_tree -- draft-tree verification.  The pages leave the
 * tree rule open ("Chains, trees and visibility": a tree needs its own
 * proposal and sampling rule); this library uses the multi-candidate form
 * of the chain rule for children drawn i.i.d. from q at their parent: at
 * node v (start: node 0, p' = p_0) try v's children in storage order; child
 * c with token t is accepted iff u[c-1]*q_v(t) < p'(t), and the walk moves
 * to c with p' = p_c; a rejected child sets p' = norm(max(0, p' - q_v)).
 * With no accepted child the final token is drawn from p' with u[N-1].
 *
 *   target_logits [B,N,V] fp32: row v scored after node v.
 *   draft_probs   [B,N,V] fp32: row v is the q that proposed v's children.
 *   node_tokens   [B,N] int32 (node 0 unused);  parent [B,N] int32 as in
 *                 spec_tree_prepare;  uniforms [B,N] fp32.
 *   accepted_len  [B] out: accepted nodes on the path.
 *   path_nodes    [B,N] out: accepted node ids, then -1.
 *   emitted       [B,N] out: accepted tokens then the final token, then -1.
 *   p_out, status_per_seq as above.  1 <= B <= 65536, 2 <= N <= 64.
 * ---------------------------------------------------------------------- */
spec_status spec_accept_sample_tree(const float* target_logits, const float* draft_probs,
                                    const int32_t* node_tokens, const int32_t* parent,
                                    const float* uniforms, int B, int N, int V,
                                    const spec_sampler* cfg, void* workspace,
                                    size_t workspace_bytes, int32_t* accepted_len,
                                    int32_t* path_nodes, int32_t* emitted, float* p_out,
                                    int32_t* status_per_seq, void* stream);

/* Copy the workspace error word to *host_err (synchronises `stream`). */
spec_status spec_workspace_error(const void* workspace, int32_t* host_err, void* stream);

/* ------------------------------------------------------------------------
 * spec_kv_commit -- keep the verified states after acceptance.
 * "Speculative Decoding" (atlas), "Committed tokens versus cached states":
 * the states of accepted proposals are kept and the rejected suffix removed;
 * the correction / bonus token's KV comes with the next pass.  "Chains,
 * trees and visibility": a tree's accepted path is compacted into the next
 * logical prefix so branch states are no longer addressable.
 *
 *   k_cache, v_cache [num_pages, page_size, Hkv, D], elem_bytes 2 (bf16) or
 *            4 (fp32), 16-byte aligned, updated in place (trees only).
 *   block_table [B, max_pages] int32; ctx_len [B] int32: block row j was
 *            written at cache position ctx_len[b] + j.
 *   accepted_len [B] int32: drafts accepted (0 .. R-1).
 *   path     [B, R] int32 (NULL: a chain, nothing moves): the accepted nodes
 *            in order, exactly as spec_accept_sample_tree writes path_nodes
 *            (node 0, the anchor, is implied and not listed; entries past
 *            accepted_len[b] are ignored).  Node ids must strictly increase
 *            (a tree in storage order puts a child after its parent).  The
 *            K/V rows of path[b][k] move to position ctx_len[b] + k + 1; node
 *            0 stays at ctx_len[b].  Every row is read before any is written.
 *   parent   [B, R] int32 (nullable; only with path): the tree's parent
 *            array; when given, each path node must be a child of the one
 *            before it (the first a child of node 0).  Without it only the
 *            order is checked and the caller must pass a real root-to-node
 *            path: the compacted keys keep the rotation of their depth.
 *   new_len  [B] int32 out: ctx_len[b] + 1 + accepted_len[b], the processed
 *            length (the anchor and the accepted drafts); the pending anchor is
 *            the emitted correction / bonus token.
 *   keep_pages [B] int32 out (nullable): block-table slots still holding a
 *            valid position, ceil(new_len / page_size); later slots the block
 *            wrote may be released.
 *   status_per_seq [B] int32 out (nullable): SPEC_SEQ_BAD_TREE when
 *            accepted_len, the path or a page index it touches is out of
 *            range, or the path breaks the rules above; that sequence is left
 *            untouched and new_len = ctx_len.
 *   1 <= R <= 64, D in {64, 128}.  Device pointers, async on the stream.
 * ---------------------------------------------------------------------- */
spec_status spec_kv_commit(void* k_cache, void* v_cache, int elem_bytes, int num_pages,
                           int page_size, int Hkv, int D, const int32_t* block_table,
                           int max_pages, const int32_t* ctx_len, const int32_t* accepted_len,
                           const int32_t* path, const int32_t* parent, int B, int R,
                           int32_t* new_len,
                           int32_t* keep_pages, int32_t* status_per_seq, void* stream);

/* ------------------------------------------------------------------------
 * spec_append_block -- write the proposed block into the paged cache, keys
 * rotated for their position.  "Speculative Decoding" (atlas), "Chains, trees
 * and visibility": position ids follow depth rather than flattened storage
 * order, so tree node j is stored at slot ctx_len + j but rotated for its
 * position id ctx_len + depth(j) (spec_tree_prepare's pos_ids).  Run it before
 * spec_verify_attn, which reads block row j at position ctx_len + j.
 *
 *   k_new, v_new [B,R,Hkv,D] dtype: the block's keys before rotation and its
 *            values.
 *   q        [B,R,Hq,D] dtype (nullable): the block's queries, rotated in
 *            place at the same positions (what spec_verify_attn then reads).
 *   k_cache, v_cache [num_pages,page_size,Hkv,D] dtype: row j of sequence b is
 *            written at position ctx_len[b] + j of its page list (the key
 *            rotated, the value as given).
 *   pos_ids  [B,R] int32 (NULL: a chain, ctx_len[b] + j).
 *   rope_base > 1: pair (x_i, x_{i+D/2}) at position t is rotated by the
 *            angle t * rope_base^(-2i/D) (the split-half rotary form; the pages
 *            do not print the rotation).  Angles are formed in double precision
 *            and reduced before the fp32 sine / cosine; rows rotate in fp32 and
 *            are rounded to the cache dtype.
 *   status_per_seq [B] int32 out (nullable): SPEC_SEQ_BAD_TREE if a row's page
 *            is missing or out of range, ctx_len < 0, the block would run past
 *            the block table, or a position id is negative; such a sequence is
 *            left untouched (no row written, no query rotated).
 *   D in {64,128}, 1 <= R <= 64.  Device pointers, async on the stream.
 * ---------------------------------------------------------------------- */
spec_status spec_append_block(const void* k_new, const void* v_new, void* q, spec_dtype dtype,
                              void* k_cache, void* v_cache, int num_pages, int page_size,
                              const int32_t* block_table, int max_pages, const int32_t* ctx_len,
                              const int32_t* pos_ids, int B, int R, int Hq, int Hkv, int D,
                              float rope_base, int32_t* status_per_seq, void* stream);

/* ------------------------------------------------------------------------
 * spec_logits_penalize -- the target logits as served, in place, before
 * spec_accept_sample(_tree).  "Speculative Decoding" (atlas), "Greedy,
 * sampling and the real sampler": p must include the transformations of the
 * served sampler -- temperature, truncation, token bans and repetition
 * penalties (the first two are spec_sampler's; this call applies the others).
 * The pages give no penalty formula; the one applied is the common
 * multiplicative form: every distinct token id in a row's prefix has its logit
 * l replaced by l / penalty if l > 0, else l * penalty (once, however often it
 * occurs), in fp32; then every banned id gets -inf.  A row's prefix is the
 * sequence's history plus the block tokens in front of the row: a chain's
 * drafts 0 .. i-1 for row i, a tree node's ancestors below the anchor and the
 * node itself.  The draft distribution q is the drafter's and is not touched.
 *
 *   logits   [B,R,V] fp32, updated in place.
 *   history  [B,H] int32: tokens already in each sequence (including the
 *            pending anchor); ids outside [0, V) (e.g. -1 padding) are skipped.
 *   block_tokens chain: [B,R-1] drafts; tree: [B,R] node tokens (node 0
 *            unused).  parent [B,R] int32 for a tree, NULL for a chain.
 *   penalty  > 0 (1: none).  banned [n_banned] int32 ids, shared by every
 *            sequence (nullable when n_banned == 0).
 *   1 <= R <= 64, V <= 172032.
 * ---------------------------------------------------------------------- */
spec_status spec_logits_penalize(float* logits, int B, int R, int V, const int32_t* history,
                                 int H, const int32_t* block_tokens, const int32_t* parent,
                                 float penalty, const int32_t* banned, int n_banned,
                                 void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
