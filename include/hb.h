/*
 * hb.h — C ABI of the block-hybrid attention library (libhb.so), sm_103a.
 *
 * Block-hybrid attention, as described for arXiv 2608.06628 ("Retrofitting
 * Linear Attention into Diffusion Language Models"; gist.science technical
 * summary, "Methodology: Block-Hybrid Attention / Architecture Design";
 * pith.science review, "What carries the argument"): inside a linearized
 * layer, every query of the active denoising block gets exact bidirectional
 * softmax attention over the block and a linear-attention read of a
 * fixed-size per-head state (S, Z) that summarises every committed token
 * through the Hedgehog feature map phi(x) = [softmax(xW), softmax(-xW)].
 * A per-head scalar gate merges the two branches.
 *
 * Notation: B requests in a call, L tokens in the active block, H heads,
 * d head dimension, f width of one softmax half, F = 2f.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.      Every pointer except `cfg` is a DEVICE pointer on the current
 *              CUDA device, owned by the caller, 16-byte aligned. The library
 *              allocates nothing; the only device memory it owns is a
 *              file-scope status word per device and the fixed scratch array
 *              of hb_prefill_state_noalloc.
 * Layouts.     Row-major, outermost index first. Activations (q, k, v, o, x)
 *              are [tokens, H, d] of the activation dtype (`cfg->dtype`).
 *              W is [H, d, f] of the activation dtype. The state pool is
 *              S_pool [num_slots, H, F, d] and Z_pool [num_slots, H, F], fp32.
 *              Within a half of phi, index c < f is softmax(xW)_c and index
 *              f + c is softmax(-xW)_c.
 * Streams.     Every call is asynchronous on `stream` (a cudaStream_t; NULL is
 *              the legacy default stream). No call synchronises except
 *              hb_get_device_status.
 * Errors.      Arguments are validated on the host before anything is
 *              launched; a rejected call returns a non-zero hb_status and has
 *              no effect. batch == 0 (or n_tokens == 0) is a valid no-op.
 *              A launch failure returns HB_ERR_CUDA. Faults that only the
 *              device can see (a slot index outside [0, num_slots), a
 *              bounded wait that ran out) never trap: the affected block of
 *              work is skipped, a bit is set in the device status word, and
 *              hb_get_device_status reports it.
 * Shapes.      1 <= H <= 1024; d in {16, 32, ..., 128}; f in {8, 16, ..., 64};
 *              1 <= L <= 64.
 * Determinism. No atomics touch S, Z or outputs; repeated calls on the same
 *              inputs give bitwise-identical results.
 * Threads.     The library keeps no per-call host state; calls from several
 *              host threads are safe.
 */
#ifndef HB_H_
#define HB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* hb_stream_t; /* same object as cudaStream_t */

typedef enum hb_status {
  HB_OK = 0,
  HB_ERR_INVALID_ARG = 1,       /* null pointer, negative size, bad enum     */
  HB_ERR_UNSUPPORTED_SHAPE = 2, /* H, d, f or L outside the supported set    */
  HB_ERR_MISALIGNED = 3,        /* a pointer is not 16-byte aligned          */
  HB_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed      */
  HB_ERR_DEVICE_BOUNDS = 5,     /* device saw a slot index out of range      */
  HB_ERR_TIMEOUT = 6,           /* a bounded device-side wait ran out        */
  HB_ERR_WORKSPACE = 7          /* workspace too small for the request       */
} hb_status;

typedef enum hb_dtype {
  HB_DTYPE_BF16 = 0, /* activations and W in bfloat16, fp32 arithmetic      */
  HB_DTYPE_FP32 = 1  /* everything fp32 (accuracy mode)                      */
} hb_dtype;

/*
 * Merge of the two branches for query i of head h (s_ij = scale * q_i.k_j,
 * sums over the L block tokens j; num_i = phi(q_i)^T S, den_i = phi(q_i)^T Z):
 *
 * HB_MERGE_SHARED_NORM — the pages' form (gist.science technical summary,
 *   merging bullet: one shared normaliser and a learned scalar gate;
 *   pith.science review, comment on the Section 3.1 out(q) equation: the
 *   gate w = sigmoid(alpha_h) scales only the softmax numerator and
 *   denominator):
 *       o_i = (w sum_j e^{s_ij} v_j + num_i) / (w sum_j e^{s_ij} + den_i)
 *   evaluated in a rescaled form that cannot overflow.
 * HB_MERGE_CONVEX — a convex blend of the two normalised branches:
 *       o_i = sigmoid(g_h) softmax_j(s_ij) v + (1 - sigmoid(g_h)) num_i / den_i
 *   and, while nothing is committed (den_i == 0), o_i = softmax_j(s_ij) v.
 */
typedef enum hb_merge {
  HB_MERGE_SHARED_NORM = 0,
  HB_MERGE_CONVEX = 1
} hb_merge;

typedef struct hb_config {
  int32_t num_heads; /* H                                   */
  int32_t head_dim;  /* d                                   */
  int32_t feat_half; /* f (F = 2f)                          */
  int32_t block_len; /* L                                   */
  int32_t dtype;     /* hb_dtype                            */
  int32_t merge;     /* hb_merge                            */
  float scale;       /* block softmax scale; 0 => 1/sqrt(d) */
} hb_config;

/*
 * hb_feature_map — phi(x) = [softmax(x W_h), softmax(-x W_h)] for every token
 * and head (gist.science technical summary, cross-block bullet; pith.science
 * review, "What carries the argument").
 *   x   [n_tokens, H, d]  activation dtype
 *   W   [H, d, f]         activation dtype
 *   phi [n_tokens, H, 2f] fp32, written
 * Each half of every output row sums to 1.
 */
hb_status hb_feature_map(const hb_config* cfg, int64_t n_tokens, const void* x,
                         const void* W, float* phi, hb_stream_t stream);

/*
 * hb_block_attend — one denoising step of a block-hybrid layer for `batch`
 * requests (gist.science technical summary, within-block, cross-block,
 * state-compression and merging bullets; pith.science review, "What carries
 * the argument": the cross-block read costs O(Fd) per query whatever the
 * prefix length).
 *   slot_idx     [batch] int32: request b reads state slot slot_idx[b]
 *   q, k, v      [batch, L, H, d] activation dtype: the active block
 *   S_pool       [num_slots, H, F, d] fp32, read only
 *   Z_pool       [num_slots, H, F] fp32, read only
 *   W            [H, d, f] activation dtype: the feature map of the queries
 *                (only phi(q) is formed here, so a state built with a
 *                separate key map by hb_commit_block / hb_prefill_state is
 *                read correctly)
 *   gate_logits  [H] fp32: alpha_h (SHARED_NORM) or g_h (CONVEX)
 *   o            [batch, L, H, d] activation dtype, written
 * A request whose slot is out of range gets no output written and sets
 * HB_ERR_DEVICE_BOUNDS in the status word.
 */
hb_status hb_block_attend(const hb_config* cfg, int32_t batch,
                          const int32_t* slot_idx, const void* q,
                          const void* k, const void* v, const float* S_pool,
                          const float* Z_pool, int32_t num_slots,
                          const void* W, const float* gate_logits, void* o,
                          hb_stream_t stream);

/*
 * hb_state_to_bf16 — write the bf16 copy of the listed slots' S that
 * hb_block_attend_s16 reads: S16[slot] = round-to-nearest bf16 of S[slot].
 * Nothing keeps the copy in step with the fp32 master by itself. These calls
 * change a slot's master and leave its copy stale: hb_commit_block,
 * hb_block_attend_commit (committing requests), hb_prefill_state,
 * hb_prefill_state_noalloc, hb_prefill_attend, hb_state_copy (destination
 * slots) and hb_state_zero. After any of them, call hb_state_to_bf16 for the
 * slots it changed before the next hb_block_attend_s16 on them; a missed
 * refresh gives outputs computed from the old state. Z needs no copy.
 *   slot_idx  [batch] int32, device
 *   S_pool    [num_slots, H, F, d] fp32, read
 *   S16_pool  [num_slots, H, F, d] bf16, written for the listed slots only
 * A slot outside [0, num_slots) is skipped and flagged as HB_ERR_DEVICE_BOUNDS.
 */
hb_status hb_state_to_bf16(const hb_config* cfg, int32_t batch,
                           const int32_t* slot_idx, const float* S_pool,
                           void* S16_pool, int32_t num_slots,
                           hb_stream_t stream);

/*
 * hb_block_attend_s16 — hb_block_attend reading the bf16 copy of S written
 * by hb_state_to_bf16 instead of the fp32 pool. The state contraction takes
 * S as bf16 operands rounded to nearest in either case, so the output is
 * bit-identical to hb_block_attend's on the fp32 states the copy was made
 * from, while each (request, head) reads 32 KiB of state instead of 64.
 * Production shape only (bf16, d = 128, f = 64, L = 32 or 16); any other shape
 * returns HB_ERR_UNSUPPORTED_SHAPE.
 *   S16_pool  [num_slots, H, F, d] bf16, read only
 *   Z_pool    [num_slots, H, F] fp32, read only (the master's Z)
 *   other arguments as in hb_block_attend.
 */
hb_status hb_block_attend_s16(const hb_config* cfg, int32_t batch,
                              const int32_t* slot_idx, const void* q,
                              const void* k, const void* v,
                              const void* S16_pool, const float* Z_pool,
                              int32_t num_slots, const void* W,
                              const float* gate_logits, void* o,
                              hb_stream_t stream);

/*
 * hb_state_to_fp8 — write an fp8 (e4m3) copy of the listed slots' S with one
 * scale per (slot, head), for hb_block_attend_s8 (gist.science technical
 * summary, state-compression bullet: a fixed-size state read at every step;
 * the copy is this library's layout, not the pages'). For each listed slot
 * and head: scale = max|S| / 448 in fp32 (rounded to nearest; 448 is the
 * largest finite e4m3 value) and code[i][j] = e4m3(S[i][j] / scale), the
 * quotient rounded to nearest in fp32 and then to the nearest e4m3 value
 * (ties to even, saturating at +-448); a head whose S is all zero gets
 * scale 0 and zero codes. The same staleness rule as hb_state_to_bf16
 * applies: every call listed there leaves the fp8 copy stale too.
 *   slot_idx    [batch] int32, device
 *   S_pool      [num_slots, H, F, d] fp32, read
 *   S8_pool     [num_slots, H, F, d] uint8 codes, written for listed slots
 *   scale_pool  [num_slots, H] fp32, written for listed slots
 * A slot outside [0, num_slots) is skipped and flagged as HB_ERR_DEVICE_BOUNDS.
 */
hb_status hb_state_to_fp8(const hb_config* cfg, int32_t batch,
                          const int32_t* slot_idx, const float* S_pool,
                          void* S8_pool, float* scale_pool, int32_t num_slots,
                          hb_stream_t stream);

/*
 * hb_block_attend_s8 — hb_block_attend reading the fp8 copy written by
 * hb_state_to_fp8: each (request, head) reads 16 KiB of state instead of 64.
 * The output is the attend on the dequantised state S' = scale * code (the
 * codes enter the state contraction exactly, as f16, with phi(q) as f16, and
 * the scale multiplies the linear read), so it differs from hb_block_attend's
 * by the copy's rounding: at the pages' shapes about 2e-3 of the output's
 * range, inside the 1e-2 bound of the bf16 outputs. Z is read from the fp32
 * pool. Production shape only (bf16, d = 128, f = 64, L = 32 or 16); any
 * other shape returns HB_ERR_UNSUPPORTED_SHAPE.
 *   S8_pool     [num_slots, H, F, d] uint8 codes, read only
 *   scale_pool  [num_slots, H] fp32, read only
 *   Z_pool      [num_slots, H, F] fp32, read only (the master's Z)
 *   other arguments as in hb_block_attend.
 */
hb_status hb_block_attend_s8(const hb_config* cfg, int32_t batch,
                             const int32_t* slot_idx, const void* q,
                             const void* k, const void* v, const void* S8_pool,
                             const float* scale_pool, const float* Z_pool,
                             int32_t num_slots, const void* W,
                             const float* gate_logits, void* o,
                             hb_stream_t stream);

/*
 * hb_block_attend_commit — hb_block_attend followed, for the requests whose
 * block is finished, by hb_commit_block of that same block, in one pass over
 * the state (gist.science technical summary, state-compression bullet: the
 * state is updated only when a block is committed). Request b's output is
 * computed against its state as it was before the call; then, if
 * commit[b] != 0, S and Z of slot_idx[b] receive sum_t phi(k_t) v_t^T and
 * sum_t phi(k_t) over this block's k, v. The state tile is read from HBM once
 * and written back once, instead of being read again by a separate commit.
 *   commit   [batch] int32, device: nonzero = this request commits its block
 *   S_pool, Z_pool  read for every request, written for committing ones
 *   W        one feature map for both the queries and the committed keys
 *   other arguments as in hb_block_attend.
 * A committing request's slot must not be read by any other request of the
 * same call (distinct slots, as in hb_commit_block).
 */
hb_status hb_block_attend_commit(const hb_config* cfg, int32_t batch,
                                 const int32_t* slot_idx, const void* q,
                                 const void* k, const void* v, float* S_pool,
                                 float* Z_pool, int32_t num_slots,
                                 const void* W, const float* gate_logits,
                                 const int32_t* commit, void* o,
                                 hb_stream_t stream);

/*
 * hb_block_attend_commit_layers — the fused step (hb_block_attend_commit) of
 * n_layers independent linearized layers in one launch. The pages' model
 * linearizes several attention layers (gist.science, "How They Did It: The
 * Two-Stage Upgrade", Stage 1: six of its twenty attention layers are
 * replaced; pith.science, "Extended reading notes", Core claim), each with
 * its own feature map, gate and states. In a forward pass the layers run one
 * after another; their steps are independent only when their inputs are
 * ready together (micro-batches at different layers, or a stack of
 * synthetic layers), and then one launch spreads all of them over the GPU
 * instead of one launch per layer.
 *   n_layers     >= 1; the call holds n_layers x batch requests, request
 *                r = l * batch + b being layer l's request b
 *   slot_idx     [n_layers * batch] int32: each request's slot in the one
 *                pool shared by the layers (the caller keeps them apart)
 *   q, k, v, o   [n_layers * batch, L, H, d] activation dtype
 *   S_pool, Z_pool  as in hb_block_attend_commit
 *   W            [n_layers, H, d, f]: layer l's feature maps
 *   gate_logits  [n_layers, H] fp32: layer l's gates
 *   commit       [n_layers * batch] int32, or NULL: attend only (the pools
 *                are then only read)
 * Equal, request by request, to n_layers calls of hb_block_attend_commit
 * (hb_block_attend when commit is NULL) on each layer's slice; a committing
 * request's slot must not be read by any other request of the call. The
 * production shape (bf16, d = 128, f = 64, L = 32 or 16) runs as one
 * launch; other shapes run as one call per layer, in layer order.
 */
hb_status hb_block_attend_commit_layers(const hb_config* cfg, int32_t n_layers,
                                        int32_t batch, const int32_t* slot_idx,
                                        const void* q, const void* k, const void* v,
                                        float* S_pool, float* Z_pool,
                                        int32_t num_slots, const void* W,
                                        const float* gate_logits,
                                        const int32_t* commit, void* o,
                                        hb_stream_t stream);

/*
 * hb_block_attend_commit_s16 — hb_block_attend_commit for a pool that keeps,
 * beside every slot's fp32 master S, the bf16 copy hb_state_to_bf16 writes
 * (gist.science technical summary, state-compression bullet: the state is
 * read every step and changes only when a block is committed; pith.science
 * review, "What carries the argument": the read is O(Fd) per query). A
 * request that does not commit reads its slot's copy (32 KiB per head
 * instead of 64); a committing request reads the master, adds its block, and
 * stores the new master and the new copy (round to nearest), so the copy
 * stays in step without a separate hb_state_to_bf16 pass. While every listed
 * slot's copy is the round-to-nearest of its master on entry, o, S_pool and
 * Z_pool come out bit-identical to hb_block_attend_commit's on the masters.
 * Production shape only (bf16, d = 128, f = 64, L = 32 or 16); any other shape
 * returns HB_ERR_UNSUPPORTED_SHAPE.
 *   S_pool    [num_slots, H, F, d] fp32 masters: read for committing
 *             requests and written for them
 *   S16_pool  [num_slots, H, F, d] bf16 copies: read for the others,
 *             written for committing requests
 *   other arguments as in hb_block_attend_commit.
 */
hb_status hb_block_attend_commit_s16(const hb_config* cfg, int32_t batch,
                                     const int32_t* slot_idx, const void* q,
                                     const void* k, const void* v, float* S_pool,
                                     void* S16_pool, float* Z_pool,
                                     int32_t num_slots, const void* W,
                                     const float* gate_logits,
                                     const int32_t* commit, void* o,
                                     hb_stream_t stream);

/*
 * hb_prefill_attend — a prompt processed block by block with block-hybrid
 * attention, so that every prompt token also gets its output (gist.science
 * technical summary, "Methodology: Block-Hybrid Attention / Architecture
 * Design": exact softmax inside the active block, linear attention over the
 * committed blocks through S and Z, which change only when a block is
 * committed). The prompt is cut into seq_len / L blocks; block j is the
 * active block against the state of blocks 0 .. j - 1 (plus the slot's
 * existing state when accumulate = 1) and is then committed. This library's
 * reading of prefill with outputs: the pages run this form when they train
 * the layers against the softmax teacher; they give no separate prefill
 * formula.
 *   slot_idx     [batch] int32, device: request b's state slot (distinct)
 *   q, k, v      [batch, seq_len, H, d] activation dtype: the prompts
 *   seq_len      prompt length, a multiple of L (every prompt has it)
 *   S_pool, Z_pool  the slots' states: zeroed first when accumulate = 0,
 *                continued from when accumulate = 1; hold the whole
 *                prompt's commit at the end
 *   W            one feature map for both queries and keys
 *   gate_logits  as in hb_block_attend
 *   o            [batch, seq_len, H, d] activation dtype, written
 * Asynchronous on `stream` and graph-capturable (a state reset when
 * accumulate = 0, then one launch in which each (request, head) walks its
 * blocks in order with the state kept on chip; other shapes take one attend
 * and one commit launch per block). seq_len not a multiple of L returns
 * HB_ERR_INVALID_ARG; a bad slot is flagged as in hb_block_attend.
 */
hb_status hb_prefill_attend(const hb_config* cfg, int32_t batch,
                            const int32_t* slot_idx, const void* q,
                            const void* k, const void* v, int64_t seq_len,
                            float* S_pool, float* Z_pool, int32_t num_slots,
                            const void* W, const float* gate_logits,
                            int32_t accumulate, void* o, hb_stream_t stream);

/*
 * hb_block_attend_ex — hb_block_attend, or with `commit` hb_block_attend_commit,
 * for layers with grouped-query heads and/or separate query and key feature
 * maps. The pages name "feature map matrices W" of a layer without saying
 * whether queries and keys share one (gist.science technical summary,
 * "Retrofitting Strategy", stage 1 bullet) and say nothing of head counts;
 * this call takes both readings: query head h uses the query map Wq[h] and
 * reads key/value head g = h / (H / H_kv), whose keys, values and state
 * (S, Z) it shares with the other query heads of its group, the state being
 * built with the key map Wk[g] (the read phi_Wq(q)^T S of pith.science,
 * "What carries the argument", with S = sum_t phi_Wk(k_t) v_t^T).
 *   num_kv_heads H_kv, which divides H = cfg->num_heads
 *   q, o         [batch, L, H, d] activation dtype (o written)
 *   k, v         [batch, L, H_kv, d] activation dtype
 *   S_pool       [num_slots, H_kv, F, d] fp32; Z_pool [num_slots, H_kv, F] fp32
 *   Wq           [H, d, f] the queries' map;  Wk [H_kv, d, f] the keys' map
 *                (used only by commits; may be NULL when commit is NULL)
 *   gate_logits  [H] fp32, per query head
 *   commit       [batch] int32 or NULL: with it, requests with commit[b] != 0
 *                then fold their block's k, v (key/value heads, map Wk) into
 *                their slot; outputs use the state as it was before the call
 * With H_kv = H and Wk == Wq (the same pointer) this is exactly
 * hb_block_attend(_commit). Otherwise the attend runs first (one launch, the
 * tensor-core kernel for the production shape when H / H_kv divides 512)
 * and the commit second (one launch), in stream order.
 */
hb_status hb_block_attend_ex(const hb_config* cfg, int32_t num_kv_heads,
                             int32_t batch, const int32_t* slot_idx,
                             const void* q, const void* k, const void* v,
                             float* S_pool, float* Z_pool, int32_t num_slots,
                             const void* Wq, const void* Wk,
                             const float* gate_logits, const int32_t* commit,
                             void* o, hb_stream_t stream);

/*
 * hb_prefill_attend_ex — hb_prefill_attend with grouped-query heads and/or a
 * separate key map, in the same reading as hb_block_attend_ex: block j of
 * query head h attends (map Wq[h]) to the state of key/value head
 * h / (H / H_kv) left by blocks 0 .. j - 1, then every key/value head's state
 * takes the block's k, v through Wk.
 *   q, o [batch, seq_len, H, d]; k, v [batch, seq_len, H_kv, d]
 *   S_pool, Z_pool  [num_slots, H_kv, ...]; Wq [H, d, f]; Wk [H_kv, d, f]
 *   other arguments as in hb_prefill_attend.
 * With H_kv = H the production shape runs one launch whatever the maps (the
 * key map is kept on chip beside the state); grouped heads take an attend
 * and a commit launch per block.
 */
hb_status hb_prefill_attend_ex(const hb_config* cfg, int32_t num_kv_heads,
                               int32_t batch, const int32_t* slot_idx,
                               const void* q, const void* k, const void* v,
                               int64_t seq_len, float* S_pool, float* Z_pool,
                               int32_t num_slots, const void* Wq, const void* Wk,
                               const float* gate_logits, int32_t accumulate,
                               void* o, hb_stream_t stream);

/*
 * hb_commit_block — fold a finished block into the state (gist.science
 * technical summary, state-compression bullet: the states change only when a
 * block is committed; pith.science review, "What carries the argument":
 * S_n = S_{n-1} + sum_t phi(k_t) v_t^T, Z_n = Z_{n-1} + sum_t phi(k_t)).
 *   slot_idx [batch] int32, distinct slots (two requests writing one slot race)
 *   k, v     [batch, L, H, d] activation dtype: the committed block
 *   W        [H, d, f]: the feature map of the keys
 *   S_pool, Z_pool updated in place for the listed slots only.
 */
hb_status hb_commit_block(const hb_config* cfg, int32_t batch,
                          const int32_t* slot_idx, const void* k,
                          const void* v, const void* W, float* S_pool,
                          float* Z_pool, int32_t num_slots, hb_stream_t stream);

/*
 * hb_prefill_state — ingest prompts as committed context (gist.science
 * technical summary, "Methodology: Block-Hybrid Attention / Architecture
 * Design", state-compression bullet: the state summarises all previously
 * committed blocks, and a prompt precedes the first generated block;
 * pith.science review, "What carries the argument": S and Z are plain sums
 * over the committed tokens). The same sums as hb_commit_block over every
 * prompt token; the sums are order-free, so the chunking does not change the
 * result.
 *   k, v        [total_tokens, H, d] activation dtype, requests packed
 *               back to back (NULL allowed when total_tokens == 0)
 *   cu_seqlens  [batch + 1] int64, device: request b owns token rows
 *               [cu_seqlens[b], cu_seqlens[b+1]); a request whose rows fall
 *               outside [0, total_tokens) is skipped and flagged as
 *               HB_ERR_DEVICE_BOUNDS
 *   max_seqlen  host upper bound on any request's length (sizes the grid).
 *               A request longer than max_seqlen, or with a negative length,
 *               is skipped (its slot is left untouched) and flagged as
 *               HB_ERR_DEVICE_BOUNDS
 *   accumulate  0: S, Z of each slot are overwritten with the prompt's sums;
 *               1: the sums are added to what the slot holds
 *   workspace   device scratch of hb_prefill_workspace_size() bytes or more
 *               (NULL allowed when that size is 0); contents need not be
 *               initialised and are clobbered
 */
hb_status hb_prefill_state(const hb_config* cfg, int32_t batch,
                           const int32_t* slot_idx, const void* k,
                           const void* v, int64_t total_tokens,
                           const int64_t* cu_seqlens, int64_t max_seqlen, const void* W, float* S_pool,
                           float* Z_pool, int32_t num_slots,
                           int32_t accumulate, void* workspace,
                           size_t workspace_bytes, hb_stream_t stream);

/* Bytes of workspace hb_prefill_state needs for this shape (may be 0).
 * Returns 0 as well for arguments hb_prefill_state would reject. */
size_t hb_prefill_workspace_size(const hb_config* cfg, int32_t batch,
                                 int64_t max_seqlen);

/*
 * hb_prefill_state_noalloc — hb_prefill_state for callers that cannot call
 * cudaMalloc: a plug-in whose host engine owns all device memory and gives it
 * no allocator, or a latency-critical serving loop where an allocation could
 * synchronise the device. The pages have no counterpart; it is a deployment
 * variant of hb_prefill_state with the same arguments, meaning and result,
 * minus the workspace.
 *   Scratch   the split partial sums live in one file-scope device array of
 *             HB_PREFILL_NOALLOC_SCRATCH_BYTES (10 MiB). Every GPU that loads
 *             the library holds it until the process exits. The call itself
 *             allocates nothing (no cudaMalloc, no allocating library call).
 *   Limit     a shape whose hb_prefill_workspace_size() exceeds that size is
 *             rejected with HB_ERR_WORKSPACE before anything is launched. For
 *             d = 128, f = 64 in bf16 the need never exceeds ~9.8 MB; every
 *             other shape needs none.
 *   Set-up    the first call on a device that needs scratch looks up the
 *             array's device address (with that device current) and caches
 *             it; make that first call before any stream capture. Under
 *             CUDA's lazy module loading (the default), that look-up may be
 *             what loads the library's device code on that device, and with
 *             it reserves the 10 MiB array there: the one-time device memory
 *             cost falls on that first call, not on loading the library.
 *   Sharing   every call on a device uses the same array. Calls whose kernels
 *             overlap on the GPU (different streams, no ordering between
 *             them) race on it; order them on one stream or with events.
 *             Nothing in the array needs to start at zero: each call writes
 *             every partial it reads back.
 */
#define HB_PREFILL_NOALLOC_SCRATCH_BYTES (10u * 1024u * 1024u)
hb_status hb_prefill_state_noalloc(const hb_config* cfg, int32_t batch,
                                   const int32_t* slot_idx, const void* k,
                                   const void* v, int64_t total_tokens,
                                   const int64_t* cu_seqlens, int64_t max_seqlen,
                                   const void* W, float* S_pool, float* Z_pool,
                                   int32_t num_slots, int32_t accumulate,
                                   hb_stream_t stream);

/*
 * hb_state_zero — clear S and Z of the listed slots: the state of a request
 * with no committed block yet (gist.science technical summary, state-
 * compression bullet: the state summarises all previously committed blocks,
 * so with none it is the empty sum, S = 0 and Z = 0; pith.science review,
 * "What carries the argument": S_0 = 0, Z_0 = 0 before the first commit).
 * Used for a new request with no prompt, or a finished request's slot being
 * recycled.
 *   slot_idx  [batch] int32, device; a slot outside [0, num_slots) is skipped
 *             and flagged as HB_ERR_DEVICE_BOUNDS
 */
hb_status hb_state_zero(const hb_config* cfg, int32_t batch,
                        const int32_t* slot_idx, float* S_pool, float* Z_pool,
                        int32_t num_slots, hb_stream_t stream);

/*
 * hb_state_copy — copy S and Z of slot src_slot[b] to slot dst_slot[b] for
 * every b < batch, within one pool. The state is a request's whole summary of
 * its committed blocks (gist.science technical summary, state-compression
 * bullet), so this snapshots a request before it is preempted, restores it,
 * or forks it into a second request with the same history.
 *   src_slot, dst_slot [batch] int32, device. Destinations must be distinct,
 *                    and no slot may be both a source and a destination of
 *                    one call (those copies would race); src == dst is a no-op
 *   S_pool, Z_pool   [num_slots, H, F, d] and [num_slots, H, F] fp32
 * A pair with a slot outside [0, num_slots) is skipped and flagged as
 * HB_ERR_DEVICE_BOUNDS.
 */
hb_status hb_state_copy(const hb_config* cfg, int32_t batch,
                        const int32_t* src_slot, const int32_t* dst_slot,
                        float* S_pool, float* Z_pool, int32_t num_slots,
                        hb_stream_t stream);

/*
 * hb_softmax_kv_attend — the full-prefix softmax attention that block-hybrid
 * attention replaces (arXiv abstract: every denoising step still attends to
 * all previous blocks; gist.science technical summary, problem statement).
 * Comparison path only. Query i of request b attends, unmasked, to the
 * request's P_b cached keys followed by the L keys of its active block.
 *   k_cache, v_cache [total_prefix, H, d] activation dtype, packed per request
 *                    (NULL allowed when total_prefix == 0)
 *   cu_prefix        [batch + 1] int64, device (P_b = cu_prefix[b+1]-cu_prefix[b]);
 *                    rows outside [0, total_prefix) are flagged, never read
 *   max_prefix       host upper bound on any P_b (sizes the grid); a request
 *                    with P_b > max_prefix or P_b < 0 gets no output written
 *                    and is flagged as HB_ERR_DEVICE_BOUNDS
 *   q, k, v          [batch, L, H, d]; o [batch, L, H, d] written
 *   workspace        device scratch of hb_softmax_kv_workspace_size() bytes
 */
hb_status hb_softmax_kv_attend(const hb_config* cfg, int32_t batch,
                               const void* k_cache, const void* v_cache,
                               int64_t total_prefix, const int64_t* cu_prefix,
                               int64_t max_prefix,
                               const void* q, const void* k, const void* v,
                               void* o, void* workspace,
                               size_t workspace_bytes, hb_stream_t stream);

/* Bytes of workspace hb_softmax_kv_attend needs for this shape (may be 0). */
size_t hb_softmax_kv_workspace_size(const hb_config* cfg, int32_t batch,
                                    int64_t max_prefix);

/*
 * hb_softmax_kv_attend_paged — hb_softmax_kv_attend over a paged KV cache
 * (PagedAttention, Kwon et al., SOSP 2023; gist.science technical summary,
 * "Key Contributions", implementation bullet: the method's serving kernel
 * keeps the fixed-size state next to paged KV caches). Comparison path only;
 * the same output as the packed call on the same tokens.
 *   k_pages, v_pages [num_pages, page_tokens, H, d] activation dtype, a pool
 *                    shared by all requests (NULL allowed when num_pages == 0)
 *   page_table       [batch, max_pages] int32, device: row b lists request b's
 *                    pages in token order; cached token t of request b is
 *                    row t % page_tokens of page page_table[b][t / page_tokens].
 *                    Only the first ceil(P_b / page_tokens) entries of a row
 *                    are read (NULL allowed when max_pages == 0)
 *   prefix_len       [batch] int32, device: P_b, the request's cached tokens.
 *                    Slots of its last page past token P_b - 1 are never
 *                    read into a sum and may hold anything, NaN included
 *   max_prefix       host upper bound on any P_b (sizes the grid), < 2^31
 *   q, k, v          [batch, L, H, d]; o [batch, L, H, d] written
 *   workspace        device scratch of hb_softmax_kv_workspace_size(cfg,
 *                    batch, max_prefix) bytes suffices
 * A request with P_b < 0, P_b > max_prefix, more than max_pages pages, or a
 * page id outside [0, num_pages) among the pages it reads gets no output
 * written and is flagged as HB_ERR_DEVICE_BOUNDS; no page outside the pool
 * is ever read. bf16 with d = 128, L = 32 and page_tokens a multiple of 32
 * takes the TMA kernel; every other case a plain kernel.
 */
hb_status hb_softmax_kv_attend_paged(const hb_config* cfg, int32_t batch,
                                     const void* k_pages, const void* v_pages,
                                     int64_t num_pages, int32_t page_tokens,
                                     const int32_t* page_table, int32_t max_pages,
                                     const int32_t* prefix_len, int64_t max_prefix,
                                     const void* q, const void* k, const void* v,
                                     void* o, void* workspace,
                                     size_t workspace_bytes, hb_stream_t stream);

/*
 * hb_get_device_status — synchronise `stream`, then read and clear the
 * current device's status word. Returns HB_OK when no device-side fault was
 * recorded since the last call, else HB_ERR_DEVICE_BOUNDS or HB_ERR_TIMEOUT
 * (bounds first when both were seen), or HB_ERR_CUDA if the synchronisation
 * itself failed.
 */
hb_status hb_get_device_status(hb_stream_t stream);

/*
 * hb_set_wait_limit — fault injection for tests of the timeout path; the
 * pages have no counterpart. Every wait inside the unit pipeline of the
 * attend kernels (hb_block_attend, hb_block_attend_s16,
 * hb_block_attend_commit, hb_block_attend_commit_s16, hb_prefill_attend)
 * gives up after `cycles` SM clocks, records HB_ERR_TIMEOUT in the device
 * status word, and the kernel winds down: it hands back no stage whose
 * copies were not seen to land, and before exiting it waits, with the
 * default limit, for the copies and tensor-core work it already issued.
 * Work after the first wait that ran out is skipped, so outputs and states
 * of that call are unspecified. cycles = 0 restores the default, 2^32 clocks
 * (about 2 s), which no wait of a healthy call comes near; values above 2^40
 * are clamped. Process-wide; it applies to launches made after the call and
 * is not meant for production use. The other kernels keep the default.
 */
hb_status hb_set_wait_limit(uint64_t cycles);

/* Static, NUL-terminated description of a status code. */
const char* hb_status_string(hb_status status);

#ifdef __cplusplus
}
#endif

#endif /* HB_H_ */
