/*
 * msa.h — C ABI of libmsa.so: the decode hot path of MiniMax Sparse Attention
 * (MSA) on one GB300 GPU (sm_103a).
 *
 * The method (sources named by page title and section):
 *   "MiniMax M3 vLLM サポート：1M トークンマルチモーダル推論の Day-0 サービング"
 *   (agentlenshq.com), section "MSA 実行プロセス": every query token goes
 *   through 1) block scoring by a small index head, 2) top-k block selection
 *   with local_blocks=1, 3) sparse GQA with online softmax over the selected
 *   blocks only; section "KV キャッシュ統合": the KV data stays an ordinary
 *   paged cache; section "EAGLE3 を用いた投機的デコード": a decode-only split-K
 *   path serves a unified decode_query_len (speculative verification).
 *   "MiniMax-M3.1-Flash Day-0 対応" (aisoku.org), section "MSAの仕組み":
 *   128-token blocks, top blocks plus the most recent block, at most 2,048 keys
 *   per query; section "何が新しいか": NVFP4 KV cache.
 *   "vLLM、AMD Instinct MI355X上でMiniMax M3のボトルネック最適化手法を公開"
 *   (news.ainew.jp), question 1: 64 query heads, 4 KV heads, 4 index heads;
 *   question 2: the indexer covers all draft positions of a request per key
 *   load and drops the positive score scale; question 5: a keys-only index
 *   cache sits beside the K/V cache.
 *
 * Conventions shared by every entry point:
 *   - Pointers named in a struct or argument list are DEVICE pointers unless
 *     the comment says "host". All memory is owned by the caller; the library
 *     allocates nothing and keeps no pointer after a call returns.
 *   - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream). Only msa_read_device_flags
 *     synchronises. The launching calls may be captured into a CUDA graph
 *     (they allocate nothing, never synchronise and read no device memory on
 *     the host); a replay reruns them with the captured arguments.
 *   - Cross-layer selection reuse ("vLLM、AMD Instinct MI355X上で…", question 3:
 *     adjacent sparse layers pick nearly the same blocks, so one layer's top-k
 *     decision serves the layers after it, which also write no index keys):
 *     a reusing layer calls msa_kv_insert_quant with idx_k_new = NULL and
 *     msa_sparse_gqa_decode with the source layer's `selected` (logical block
 *     ids, valid with the reusing layer's own block table).
 *   - Host-side validation runs before any launch. A status other than MSA_OK
 *     means nothing was launched (MSA_ERR_CUDA: a launch was attempted and the
 *     CUDA runtime reported an error).
 *   - Inputs that only the device can check (page ids in the block table,
 *     selected block ids, context lengths, cache slots) are checked by the
 *     kernels: an offending block or token is skipped and a bit is OR-ed into
 *     `*dev_flags` (a caller-owned device uint32 that the caller zeroes). No
 *     kernel traps, and every wait inside a kernel is bounded in time.
 *   - Shapes: B batch, Q query positions per request (decode_query_len), H
 *     query heads, G KV heads, I index heads (I == G), D head_dim (128),
 *     BS block size (128), P pages, NB max_blocks_per_seq, K topk.
 *     Query j of request b sits at position p = seq_lens[b] - Q + j; its
 *     local block is p / BS.
 *   - The dispatch record (msa_get_last_dispatch) is thread-local and names
 *     the kernel variant and launch shape that actually ran.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSA_ABI_VERSION 2

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
  MSA_ERR_UNSUPPORTED = 2,   /* valid request outside what the kernels implement */
  MSA_ERR_CUDA = 3,          /* the CUDA runtime reported an error at launch */
  MSA_ERR_WORKSPACE = 4,     /* workspace null or smaller than msa_sparse_gqa_workspace_size */
  MSA_ERR_DEVICE_FLAG = 5    /* msa_read_device_flags found a kernel-reported problem */
} msa_status_t;

typedef enum {
  MSA_F32 = 0,
  MSA_BF16 = 1,
  MSA_FP8_E4M3 = 2,
  MSA_NVFP4 = 3
} msa_dtype_t;

/* Bits a kernel may OR into *dev_flags. */
#define MSA_FLAG_BAD_PAGE      0x1u  /* block_table entry outside [0, num_pages) */
#define MSA_FLAG_BAD_BLOCK     0x2u  /* selected block id beyond the query's local block */
#define MSA_FLAG_BAD_SEQLEN    0x4u  /* seq_lens[b] < q_len or > max_blocks_per_seq * BS */
#define MSA_FLAG_BAD_SLOT      0x8u  /* slot_mapping entry >= num_pages * BS */
#define MSA_FLAG_TIMEOUT       0x10u /* a bounded wait inside a kernel gave up */
#define MSA_FLAG_Q_RANGE       0x20u /* an index-query row too large for the fp16 operand path */

/* Problem shape (host struct). block_size must be 128, head_dim 128,
 * local_blocks 1, n_idx_heads == n_kv_heads, n_heads % n_kv_heads == 0,
 * 1 <= topk <= 16, 1 <= q_len <= 8. */
typedef struct {
  int32_t batch;               /* B */
  int32_t q_len;               /* Q, query positions per request */
  int32_t n_heads;             /* H */
  int32_t n_kv_heads;          /* G */
  int32_t n_idx_heads;         /* I */
  int32_t head_dim;            /* D */
  int32_t block_size;          /* BS */
  int32_t max_blocks_per_seq;  /* NB, columns of block_table and scores */
  int32_t num_pages;           /* P */
  int32_t topk;                /* K, blocks selected per (b, j, head), local block included */
  int32_t local_blocks;        /* must be 1 */
  float softmax_scale;         /* logits = softmax_scale * q.k */
} msa_dims_t;

/* Paged K/V cache of one layer (host struct holding device pointers).
 *   MSA_BF16:  k, v  = bf16 [P, G, BS, D]; k_scale = v_scale = NULL.
 *   MSA_FP8_E4M3: k, v = uint8 E4M3 codes [P, G, BS, D]; k_global, v_global =
 *              fp32 per-tensor scales (host values, > 0); value = e4m3 * global
 *              (61,440 bytes per token over 60 layers: "MiniMax-M3.1-Flash
 *              Day-0 対応", section "何が新しいか"); k_scale = v_scale = NULL.
 *   MSA_NVFP4: k, v  = uint8 [P, G, BS, D/2] E2M1 pairs, low nibble = even
 *              element; k_scale, v_scale = uint8 E4M3 [P, G, BS, D/16], one
 *              per 16 consecutive elements; k_global, v_global = fp32
 *              per-tensor scales (host values, > 0).
 *   value = e2m1 * e4m3_scale * global. 16-byte aligned pointers. */
typedef struct {
  msa_dtype_t dtype;
  void* k;
  void* v;
  void* k_scale;
  void* v_scale;
  float k_global;
  float v_global;
} msa_kv_cache_t;

/* Keys-only index cache of one layer (host struct holding device pointers).
 *   MSA_F32:      keys = fp32 [P, I, BS, D]; scale = NULL.
 *   MSA_FP8_E4M3: keys = uint8 E4M3 [P, I, BS, D]; scale = fp32 [P, I, BS],
 *                 one per (token, index head); key value = e4m3 * scale.
 *   MSA_NVFP4:    keys = uint8 [P, I, BS, D/2] E2M1 pairs (low nibble = even
 *                 element); block_scale = uint8 E4M3 [P, I, BS, D/16];
 *                 global_scale = fp32 per-tensor scale (host value, > 0);
 *                 key value = e2m1 * e4m3 * global ("MiniMax-M3.1-Flash
 *                 Day-0 対応", section "試し方": indexer_kv_dtype nvfp4).
 *   16-byte aligned pointers. */
typedef struct {
  msa_dtype_t dtype;
  void* keys;
  float* scale;
  void* block_scale;
  float global_scale;
} msa_index_cache_t;

/* ABI version of the loaded library (MSA_ABI_VERSION at build time). */
int msa_abi_version(void);

/* Human-readable name of a status. Never NULL. */
const char* msa_status_string(msa_status_t status);

/* Copies the thread-local record of the last kernel launch into buf (NUL
 * terminated, truncated to len). */
msa_status_t msa_get_last_dispatch(char* buf, size_t len);

/*
 * Cache insertion and quantisation: writes num_tokens new tokens into the
 * paged caches. The pages give the caches (paged KV, a keys-only index cache,
 * NVFP4 KV, an FP8 indexer on the roadmap) but no quantisation rule; the rule
 * implemented is:
 *   FP8 index keys: s = amax / 448 over the token's D values of that head (fp32,
 *     IEEE division), code = E4M3_RNE_satfinite(x / s); s = 0 -> codes 0.
 *   NVFP4 K/V and NVFP4 index keys: per 16 values sb = E4M3_RNE((amax16 / 6) /
 *     global), code = E2M1_RNE_satfinite(x / (sb * global)); sb == 0 -> codes 0.
 *   FP8 K/V: code = E4M3_RNE_satfinite(x / global) (fp32 IEEE division).
 *   bf16 K/V and fp32 index keys are copied.
 * k_new, v_new: bf16 [T, G, D]. idx_k_new: [T, I, D] of idx_new_dtype
 * (MSA_F32 or MSA_BF16; MSA_BF16 requires an FP8 or NVFP4 index cache), or NULL to
 * leave the index cache untouched (idx_cache may then be NULL).
 * slot_mapping: int64 [T], slot = page * BS + offset; a negative slot skips
 * the token; slot >= P * BS skips it and sets MSA_FLAG_BAD_SLOT.
 */
msa_status_t msa_kv_insert_quant(const msa_dims_t* dims, const void* k_new, const void* v_new,
                                 const void* idx_k_new, msa_dtype_t idx_new_dtype,
                                 const int64_t* slot_mapping, int32_t num_tokens,
                                 const msa_kv_cache_t* cache, const msa_index_cache_t* idx_cache,
                                 uint32_t* dev_flags, void* stream);

/* RMSNorm weights and rotary parameters of msa_qk_norm_rope_insert (host
 * struct; the weights are device fp32 [D] arrays, 16-byte aligned). */
typedef struct {
  const float* q_weight;
  const float* k_weight;
  const float* idx_q_weight;   /* may be NULL when the call has no index rows */
  const float* idx_k_weight;
  float eps;                   /* >= 0 */
  float rope_theta;            /* rotary base, > 1 */
} msa_norm_rope_t;

/*
 * The step in front of the decode path, fused: per-head RMSNorm of the query,
 * key, index-query and index-key projections, rotary position embedding, and
 * insertion of the key, V and index key into the caches ("MiniMax-M3.1-Flash
 * Day-0 対応", section "最適化と数値": QKV GEMM + norm + RoPE + KV insert;
 * "MiniMax M3 vLLM サポート：…", section "カーネル融合": QKNorm + RoPE + KV
 * insertion). The pages give no formulas; implemented (fp32, one CTA per token):
 *   norm:  y_d = x_d / sqrt(mean_d(x^2) + eps) * w_d (IEEE sqrt and division);
 *   RoPE:  for i < D/2, phi = position * rope_theta^(-2i/D) (angle in double
 *          precision), (y_i, y_{i+D/2}) <- (y_i cos - y_{i+D/2} sin,
 *          y_i sin + y_{i+D/2} cos) — all D dims, the two halves paired;
 *   the results are rounded to bf16: q_out / idx_q_out receive them, and the
 *   key and index key go through the cache quantisers of msa_kv_insert_quant
 *   (as if inserted from those bf16 values); V is inserted unchanged.
 * q: bf16 [T, H, D]; k, v: bf16 [T, G, D]; idx_q, idx_k: bf16 [T, I, D], both
 * NULL for a layer that reuses another layer's selection (then idx_q_out,
 * idx_cache and the index weights may be NULL and no index row is touched:
 * "vLLM、AMD Instinct MI355X上で…", question 3). positions: int32 [T] (the
 * token's position in its sequence). slot_mapping: as msa_kv_insert_quant.
 * q_out: bf16 [T, H, D], idx_q_out: bf16 [T, I, D] (may alias q / idx_q). The
 * index cache must be FP8 or NVFP4 (MSA_ERR_UNSUPPORTED otherwise).
 */
msa_status_t msa_qk_norm_rope_insert(const msa_dims_t* dims, const void* q, const void* k, const void* v,
                                     const void* idx_q, const void* idx_k, const int32_t* positions,
                                     const int64_t* slot_mapping, int32_t num_tokens, const msa_norm_rope_t* nr,
                                     void* q_out, void* idx_q_out, const msa_kv_cache_t* cache,
                                     const msa_index_cache_t* idx_cache, uint32_t* dev_flags, void* stream);

/*
 * Stage 1, block scoring ("MSA 実行プロセス" step 1). For every request b,
 * position j, index head g and block n < l_j (the query's local block):
 *   scores[b, j, g, n] = max over the block's 128 tokens t of s_t * (q_idx[b, j, g] . k_t)
 * with s_t the key's per-token scale (1 for fp32 and NVFP4 keys; NVFP4 keys
 * carry their block and global scales in k_t); no other scale is applied (a
 * positive constant cannot change the selection). All other
 * entries up to max_blocks_per_seq are set to -inf. All Q positions of a
 * request are computed from one load of each index key.
 * idx_q: [B, Q, I, D] in q_dtype (MSA_F32 with an MSA_F32 index cache,
 * MSA_BF16 with an MSA_FP8_E4M3 or MSA_NVFP4 one). block_table: int32 [B, NB].
 * seq_lens: int32 [B]. scores: fp32 [B, Q, I, NB].
 * With FP8 or NVFP4 keys the last eighth of the blocks is handed out to the
 * CTAs at run time from a queue in a library-owned device array: direct calls
 * take one of 64 slots in turn (at most 64 may run at once), and launches
 * captured into CUDA graphs one of 64 other slots in turn (at most 64 captured
 * launches may be in use). The CTA that finishes last resets its slot, so a
 * captured graph replays cleanly; after a launch that raised MSA_FLAG_TIMEOUT,
 * capture such a graph again before replaying it. The scores do not depend on
 * which CTA scored a block.
 */
msa_status_t msa_index_score(const msa_dims_t* dims, const void* idx_q, msa_dtype_t q_dtype,
                             const msa_index_cache_t* idx_cache, const int32_t* block_table,
                             const int32_t* seq_lens, float* scores, uint32_t* dev_flags,
                             void* stream);

/*
 * The insert of msa_kv_insert_quant and the scoring of msa_index_score in one
 * launch, for a decode step with one query position ("MSA 実行プロセス" steps
 * 0-1; "EAGLE3 を用いた投機的デコード" for the single-position case). The
 * step's new token of request b sits at position seq_lens[b] - 1, in the
 * request's local block, which the scoring never reads. That page must not be
 * a fully visible block in any other request's table; a paged allocator that
 * shares only full prefix blocks guarantees this. So the scoring warps
 * insert the B tokens before their first index page arrives, and the
 * attention call that follows sees the new K/V because it waits for the whole
 * launch.
 * k_new, v_new: bf16 [B, G, D]; idx_k_new: [B, I, D]; slot_mapping:
 * int64 [B], the new token of request b, which must equal
 *   block_table[b, (seq_lens[b] - 1) / 128] * 128 + (seq_lens[b] - 1) % 128
 * (negative: a padding request, skipped). A token whose slot is anything else
 * is skipped and raises MSA_FLAG_BAD_SLOT. idx_q and idx_k_new are fp32 with
 * an MSA_F32 index cache and bf16 with an FP8 E4M3 or NVFP4 one. q_len must be
 * 1, else MSA_ERR_UNSUPPORTED. Results are the two separate calls' results,
 * byte for byte.
 */
msa_status_t msa_insert_index_score(const msa_dims_t* dims, const void* k_new, const void* v_new,
                                    const void* idx_k_new, const int64_t* slot_mapping,
                                    const msa_kv_cache_t* cache, const void* idx_q,
                                    const msa_index_cache_t* idx_cache, const int32_t* block_table,
                                    const int32_t* seq_lens, float* scores, uint32_t* dev_flags, void* stream);

/*
 * Stage 2, block selection ("MSA 実行プロセス" step 2, local_blocks=1). For
 * every (b, j, g): order the candidates n < l_j by score (higher first, then
 * lower block id), keep the first min(K-1, l_j), add l_j, and write them in
 * ascending order followed by -1 padding: selected int32 [B, Q, G, K].
 * Scores are compared as exact fp32 values (NaN counts as -inf).
 */
msa_status_t msa_select_blocks(const msa_dims_t* dims, const float* scores, const int32_t* seq_lens,
                               int32_t* selected, uint32_t* dev_flags, void* stream);

/* Bytes of device workspace msa_sparse_gqa_decode needs for this shape. */
size_t msa_sparse_gqa_workspace_size(const msa_dims_t* dims, msa_dtype_t kv_dtype);

/*
 * Stage 3, sparse GQA decode ("MSA 実行プロセス" step 3; split-K decode path
 * of "EAGLE3 を用いた投機的デコード"). For every query head h of position j of
 * request b, with KV head g = h / (H / G), over the tokens t of the blocks in
 * selected[b, j, g, :] (entries < 0 ignored; each block id at most once per
 * row, as msa_select_blocks writes them) with t <= p:
 *   out[b, j, h] = sum_t softmax_t(softmax_scale * q . k_t) * v_t
 *   lse[b, j, h] = log sum_t exp(softmax_scale * q . k_t)
 * The work is split over the selected blocks and the partial results merged
 * with a log-sum-exp combine. K/V are read from bf16, FP8 E4M3 or NVFP4 pages
 * and dequantised in the kernel. Cache slots past a position's causal limit
 * never reach its result: their logits are masked and their V rows are zeroed
 * before the P.V product. So slots that were never written, such as the tail
 * of a request's last page, may hold any bytes, NaN patterns included.
 * With several query positions and bf16 K/V, the positions of a (request, KV
 * head) pair are attended together when there are at least three such pairs
 * for every four SMs: one CTA streams the union of their selected blocks once
 * and each position attends over its own blocks, on the tcgen05 tensor cores
 * with the 8 positions' 128 query rows in one tile. MSA_MULTIPOS_ATTENTION=union
 * or =rows in the environment (read on every call) forces that form or the
 * per-position one (=union_mma: the union form on mma.sync); all give the same
 * results within the same tolerances.
 * For bf16 K/V the environment variable MSA_BF16_ATTENTION=tcgen05, read on
 * every call, selects a tcgen05 form of the tile. It computes S^T = K.Q^T and
 * O^T = V^T.P^T with S and O in tensor memory and gives the same results
 * within the same tolerances, but it is slower at 16 heads per KV head. The
 * default is the mma.sync tile.
 * For NVFP4 K/V, when every row's cluster fits on the device at once, each
 * (request, position, KV head) row is split over a thread-block cluster of 8,
 * 4 or 2 CTAs whose partials are merged in distributed shared memory (no
 * workspace use); otherwise the selected blocks are balanced over all SMs and
 * split rows merge through the workspace. MSA_NVFP4_SPLIT=tickets, =cluster2,
 * =cluster4 or =cluster8 in the environment (read on every call) forces a
 * form; all give the same results within the same tolerances.
 * q: bf16 [B, Q, H, D]. out: bf16 [B, Q, H, D]. lse: fp32 [B, Q, H] or NULL.
 * workspace: device scratch of at least msa_sparse_gqa_workspace_size bytes
 * (B * Q * G * (topk * 8,320 + 8)), 256-byte aligned: split-K partials and one
 * tagged ticket per row. Its contents need no initialisation and are not
 * meaningful after the call; calls that overlap on the GPU must not share it.
 * Each call tags its tickets with a new epoch, but a captured CUDA graph
 * replays the epoch of its capture: after a launch that raised
 * MSA_FLAG_TIMEOUT, a ticket may keep that launch's partial count, so zero the
 * workspace (or capture again) before replaying such a graph. Direct calls
 * are unaffected.
 */
msa_status_t msa_sparse_gqa_decode(const msa_dims_t* dims, const void* q, const msa_kv_cache_t* cache,
                                   const int32_t* block_table, const int32_t* seq_lens,
                                   const int32_t* selected, void* out, float* lse, void* workspace,
                                   size_t workspace_bytes, uint32_t* dev_flags, void* stream);

/*
 * Stages 2 and 3 in one launch: the selection of msa_select_blocks, computed
 * by the attention kernel's own CTAs from the block scores (one warp per row
 * its CTA attends; the result is also written to `selected`, [B, Q, G, K]),
 * followed by the sparse GQA decode of msa_sparse_gqa_decode over it. Saves
 * the selection launch and its round trip on the latency path. Arguments as
 * msa_sparse_gqa_decode, with scores (fp32 [B, Q, I, NB], as written by
 * msa_index_score) as the input and selected as an output.
 */
msa_status_t msa_select_sparse_gqa_decode(const msa_dims_t* dims, const void* q, const msa_kv_cache_t* cache,
                                          const int32_t* block_table, const int32_t* seq_lens, const float* scores,
                                          int32_t* selected, void* out, float* lse, void* workspace,
                                          size_t workspace_bytes, uint32_t* dev_flags, void* stream);

/*
 * Allocation-free variant of msa_sparse_gqa_decode. The pages have no
 * counterpart: it exists for callers that cannot allocate device memory (a
 * process whose allocator owns all device memory, a plugin that receives only
 * its input and output buffers, tooling that must not change the device's
 * memory footprint). Same arguments and results as msa_sparse_gqa_decode,
 * without the workspace: the split-K partials go to a 64 MiB array inside the
 * library, which every GPU that loads the library holds until the process
 * exits. The first call on a device looks up that array's address (make it
 * before any stream capture on that device); so does the first call after the
 * device's context changed (after a cudaDeviceReset, for example), which
 * should also come before any capture. All calls on a device share the
 * array, so calls whose kernels overlap on the GPU race; nothing in it needs
 * to start at zero. Shapes whose workspace (msa_sparse_gqa_workspace_size:
 * B * Q * G * (topk * 8,320 + 8) bytes) exceeds 64 MiB return
 * MSA_ERR_WORKSPACE without launching. After a call that raised
 * MSA_FLAG_TIMEOUT, a captured graph of this call must be captured again
 * before it is replayed (the array cannot be zeroed from outside).
 * Calls no allocating routine.
 */
msa_status_t msa_sparse_gqa_decode_noalloc(const msa_dims_t* dims, const void* q, const msa_kv_cache_t* cache,
                                           const int32_t* block_table, const int32_t* seq_lens,
                                           const int32_t* selected, void* out, float* lse, uint32_t* dev_flags,
                                           void* stream);

/*
 * Diagnostic of the bounded waits (the pages have no counterpart). Launches
 * one thread that waits on a shared-memory barrier which nothing completes,
 * through the same bounded wait the library's kernels use; when the wait gives
 * up (after about 2 s) the kernel ORs MSA_FLAG_TIMEOUT into *dev_flags and
 * returns. No copy is in flight when it gives up, so the context stays usable:
 * a caller can check on its GPU that a kernel whose wait runs out reports an
 * error status instead of hanging. Asynchronous on `stream`.
 */
msa_status_t msa_selftest_bounded_wait(uint32_t* dev_flags, void* stream);

/* Synchronises `stream`, copies *dev_flags to *host_flags (host pointer) and
 * returns MSA_ERR_DEVICE_FLAG if any bit is set, MSA_OK otherwise. */
msa_status_t msa_read_device_flags(const uint32_t* dev_flags, uint32_t* host_flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
