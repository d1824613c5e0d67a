/*
 * qsa.h -- C ABI of the GB300 QSA indexer library (libqsa.so).
 *
 * The library computes, on one GPU, the data-parallel hot path of the QSA
 * sparse-attention indexer and a generic token-level top-k:
 *
 *   compress  block of 4 raw BF16 index keys -> one BF16 compressed key
 *   score     s[t][b] = (1/sqrt(128)) * sum_{h<4} ReLU(<q[t][h], kbar[b]>)
 *   select    best k visible blocks (ties: lower block id), ascending
 *   expand    block b -> token positions 4b..4b+3, then the 0-3 pending
 *             tokens of the incomplete block; -1 fills the rest
 *   translate position -> physical KV slot through the request's page table
 *
 * Sources, cited by page title and section:
 *  [QSA]  "SGLang Day-0 support for Qwen3.8-Flash-Next: QSA sparse attention,
 *         IndexShare MTP and HyperConnection kernel optimisations"
 *         (theainews.cc), section "Qwen sparse attention (QSA): coarse
 *         retrieval, fine attention" -- 4 query heads x 128 dims and one
 *         shared key head; every 4 raw index keys averaged in FP32,
 *         normalised and rotated at the block's first-token position into
 *         one compressed key; the score equation; the best 512 blocks
 *         expanded to 2048 token positions plus the 0-3 pending tokens (at
 *         most 2051); one BF16 compressed key per 4 tokens, stored
 *         page-aligned at full_slot/4.
 *  [TOPK] SGLang GLM-5.2 blog (aihot.virxact.com), section "Kernel
 *         Optimization / TopK-V2", Figures 2-4 -- exact top-k (runtime k up
 *         to 2048) over FP32 score rows, with the selected logical positions
 *         translated into physical KV-cache slots in the same kernel.
 *  [SMLA] "vllm-sparse-mla-blackwell" (shadowgraph.io), section "Design notes
 *         worth knowing" -- the attention consumer's only mask is
 *         index >= 0, so -1 marks an empty entry.
 *
 * Conventions shared by every call
 *  - Every pointer is a DEVICE pointer unless its name starts with h_.  The
 *    caller owns all memory; the library never allocates, frees, or keeps
 *    per-call state, and never synchronises.  Scratch comes from a caller
 *    workspace sized by the matching *_workspace_size() query.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call only enqueues work on it.
 *  - BF16 tensors are passed as `const void*` / `void*` (IEEE bfloat16, 2 B).
 *  - Fixed sizes: index head dim 128, 4 index query heads, 4 raw keys per
 *    compressed block.  Indices and slots are int32; leading dimensions are
 *    int64 element counts.  -1 is the sentinel for an empty entry.
 *  - Rows are grouped by request: rows req_row_start[r] .. req_row_start[r+1]-1
 *    (device int32 array of n_req+1 entries, non-decreasing, first entry 0)
 *    belong to request r.  Row t sees row_len[t] tokens (its position + 1):
 *    complete blocks b < row_len[t]/4 and row_len[t] mod 4 pending tokens.
 *    `max_len` is a host-side upper bound of every row_len[t]; it sizes the
 *    launch.
 *  - Paging: page_table is [n_req][ld_pt] int32 physical page ids;
 *    slot(pos) = page_table[r][pos / page_size] * page_size + pos % page_size.
 *    The compressed key of block b of request r lives in pool row
 *    slot(4b) / 4 (the page-aligned full_slot/4 address of [QSA]); the pool
 *    holds pool_rows rows of 128 BF16 and page_size must be a multiple of 4.
 *  - Errors: host-side argument checks return a negative qsa_status and
 *    enqueue nothing.  Launch failures return QSA_ERR_CUDA.  Device-side
 *    checks (a row longer than max_len, a page id or pool row out of range)
 *    skip the offending access and latch a device fault word, read with
 *    qsa_device_status().  No call traps or spins without a bound.
 */
#ifndef QSA_H_
#define QSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int qsa_status;
#define QSA_OK 0
#define QSA_ERR_INVALID_ARG (-1)        /* null pointer, negative size, misalignment */
#define QSA_ERR_UNSUPPORTED (-2)        /* k > 2048, page_size % 4 != 0, row too long */
#define QSA_ERR_WORKSPACE_TOO_SMALL (-3)
#define QSA_ERR_CUDA (-4)               /* a CUDA launch or query failed */
#define QSA_ERR_DEVICE_FAULT (-5)       /* a device-side bounds check fired */

#define QSA_HEAD_DIM 128
#define QSA_HEADS 4
#define QSA_BLOCK 4
#define QSA_MAX_K 2048

/* Human-readable name of a status code (static string). */
const char* qsa_status_string(qsa_status s);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int qsa_version(void);

/* Synchronises `stream`, reads the device fault word latched by the
 * device-side bounds checks of earlier calls, optionally clears it, and
 * returns QSA_OK or QSA_ERR_DEVICE_FAULT.  *h_bits (may be NULL) receives the
 * word: bit 0 row/page index out of range, bit 1 pool row out of range,
 * bit 2 a bounded wait expired, bit 3 inconsistent row grouping, bit 4 an
 * output row too narrow for its entries (qsa_indexshare_slots). */
qsa_status qsa_device_status(void* stream, int clear, uint32_t* h_bits);

/* ---------------------------------------------------------------------
 * Compressed index keys  ([QSA]: one compressed key per block of 4 raw index
 * keys -- their FP32 average, normalised, rotated at the position of the
 * block's first token -- kept in BF16 in a paged cache at full_slot/4).
 *
 *   raw        [n_blocks*4][128] BF16: the 4 raw index keys of each block,
 *              in token order.
 *   block_req  [n_blocks] request of each block (row of page_table).
 *   block_id   [n_blocks] block index b within its request; the block's first
 *              token is position 4b and its key goes to pool row slot(4b)/4.
 *   page_table [n_req][ld_pt]; NULL stores block i in pool row i instead.
 *   rope_base  RoPE base (10000 for the workloads here).
 *   pool       [pool_rows][128] BF16, written in place.
 *
 * Per block: m = ((k0 + k1) + k2) + k3 in FP32, times 0.25; u = m / ||m||_2
 * (u = 0 if m = 0); RoPE with rotate-half pairs (i, i+64), angle
 * 4b * rope_base^(-2i/128); rounded to BF16 (nearest even).
 * ------------------------------------------------------------------- */
qsa_status qsa_compress_keys(const void* raw, const int32_t* block_req, const int32_t* block_id,
                             int64_t n_blocks, int32_t n_req, const int32_t* page_table,
                             int64_t ld_pt, int32_t page_size, double rope_base, void* pool,
                             int64_t pool_rows, void* stream);

/* ---------------------------------------------------------------------
 * Decode key path through a per-request ring  ([QSA]: the raw index keys of
 * the incomplete block wait in a 4-slot ring per request instead of being
 * kept for the whole context; a completed block is compressed into the pool
 * at full_slot/4).
 *
 *   new_keys      [n_tok][128] BF16 raw index keys appended by this call.
 *   req_tok_start [n_req+1]: request r appends new_keys[req_tok_start[r] ..
 *                 req_tok_start[r+1]-1] at consecutive positions
 *                 req_first_pos[r], req_first_pos[r]+1, ...
 *   ring          [n_req][4][128] BF16, updated in place: slot p mod 4 holds
 *                 the raw key of position p of the request's incomplete
 *                 block (written by earlier calls).
 *   page_table, page_size, pool, pool_rows, rope_base: as qsa_compress_keys.
 *
 * Every block b that the appended positions complete (4b+3 among them) is
 * compressed exactly as qsa_compress_keys does, from its 4 raw keys (this
 * call's where present, the ring's for earlier positions), into pool row
 * slot(4b)/4; then ring slot p mod 4 takes the key of each appended
 * position p (the later ones win).  Device faults: a page id or pool row out
 * of range (bits 0, 1), bad grouping (bit 3).
 * ------------------------------------------------------------------- */
qsa_status qsa_append_keys(const void* new_keys, const int32_t* req_tok_start, const int32_t* req_first_pos,
                           int32_t n_req, void* ring, const int32_t* page_table, int64_t ld_pt,
                           int32_t page_size, double rope_base, void* pool, int64_t pool_rows, void* stream);

/* ---------------------------------------------------------------------
 * Block scores  ([QSA] score equation:
 *   s[t][b] = (1/sqrt(128)) * sum_{h=1..4} ReLU(<q[t][h], kbar[b]>)
 * over the visible compressed blocks b < row_len[t]/4).
 *
 *   q          [n_rows][4][128] BF16 index queries (already position-encoded).
 *   pool       compressed-key pool, addressed through page_table.
 *   scores     [n_rows][ld_scores] FP32 out.  Entries b < row_len[t]/4 are
 *              written; entries row_len[t]/4 <= b < n_fill are set to -inf;
 *              nothing else is touched.  ld_scores >= max_len/4.
 *   max_rows_per_req  host upper bound of the rows of any one request.
 * Products of BF16 are exact; accumulation is FP32.
 * ------------------------------------------------------------------- */
qsa_status qsa_index_scores(const void* q, const void* pool, int64_t pool_rows, int32_t n_req,
                            const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                            int32_t max_len, int32_t max_rows_per_req, const int32_t* page_table,
                            int64_t ld_pt, int32_t page_size, float* scores, int64_t ld_scores,
                            int64_t n_fill, void* stream);

/* ---------------------------------------------------------------------
 * Exact top-k over FP32 rows  ([TOPK]: a selection rather than a sort,
 * returning exactly k entries for a runtime k of at most 2048, with the
 * page-table transform to physical KV-cache slots done in the same kernel).
 *
 *   scores     [n_rows][ld] FP32.
 *   n_valid    [n_rows] candidates per row (entries 0..n_valid-1), or NULL:
 *              every row has n_max candidates.
 *   n_max      host upper bound of n_valid (<= ld).
 *   k          1..2048.
 *   page_table [.][ld_pt] or NULL (then out_slots must be NULL).
 *   row_req    [n_rows] page-table row of each row, or NULL: row t uses
 *              page-table row t.
 *   out_idx    [n_rows][k]: the k best indices in ascending order; -1 after
 *              the first min(k, n_valid) entries.
 *   out_slots  [n_rows][k] or NULL: slot(out_idx), -1 stays -1.
 * Order: larger value first; equal values by ascending index; -0 == +0; NaN
 * below every number.  The result is unique, so it is bit-exact.
 * Workspace: topk_select_workspace_size(...) bytes (4-byte aligned) hold a
 * row plan made on the device ([TOPK]: a planning kernel reads the batch's
 * lengths so that long rows get a cluster of CTAs and short rows one CTA);
 * it is used when n_max exceeds 32768 and there are more rows than half the
 * SMs.  With a smaller or no workspace every row takes the kernel chosen
 * from n_max and n_rows alone.  The size query may return 0.  With the plan,
 * the short rows run on a library-owned side stream beside the long ones
 * (forked from and joined back to `stream` with events, so the call's work
 * stays ordered on `stream`, stream capture included).
 * ------------------------------------------------------------------- */
size_t topk_select_workspace_size(int32_t n_rows, int32_t n_max, int32_t k);
qsa_status topk_select(const float* scores, int64_t ld, const int32_t* n_valid, int32_t n_rows,
                       int32_t n_max, int32_t k, const int32_t* page_table, int64_t ld_pt,
                       const int32_t* row_req, int32_t page_size, int32_t* out_idx,
                       int32_t* out_slots, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------
 * Expansion of selected blocks to token positions and KV slots  ([QSA]:
 * each kept block stands for its 4 token positions, and the 0-3 tokens of
 * the still-incomplete block are added after them; [TOPK] page-table
 * transform; [SMLA] -1 sentinel).
 *
 *   sel_blocks [n_rows][k_blk] ascending block ids, -1 only as tail padding.
 *   out_pos    [n_rows][4*k_blk+3] or NULL: 4b..4b+3 for each selected b in
 *              order, then positions 4*(row_len/4) .. row_len-1, then -1.
 *   out_slots  [n_rows][4*k_blk+3]: slot(out_pos), -1 stays -1.
 * ------------------------------------------------------------------- */
qsa_status qsa_expand_slots(const int32_t* sel_blocks, int32_t k_blk, int32_t n_req,
                            const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                            const int32_t* page_table, int64_t ld_pt, int32_t page_size,
                            int32_t* out_pos, int32_t* out_slots, void* stream);

/* ---------------------------------------------------------------------
 * One decode step in one call: the key path (qsa_append_keys: new raw index
 * keys into the rings, completed blocks compressed into the pool) followed
 * by the fused indexer (qsa_indexer_select) on the updated pool.
 *
 * Arguments as the two calls.  The positions this step appends must be the
 * rows' own tokens or earlier, i.e. the compressed blocks the scorer reads
 * may include the ones completed here.  The scorer reads no pool row the key
 * path writes before that write is done; scorer CTAs whose key range ends
 * before block req_first_pos[r]/4 do not wait for the key path at all (the
 * launch is ordered with programmatic dependent launch).  Results equal the
 * two calls made one after the other.
 * ------------------------------------------------------------------- */
qsa_status qsa_decode_step(const void* new_keys, const int32_t* req_tok_start, const int32_t* req_first_pos,
                           void* ring, double rope_base, const void* q, void* pool, int64_t pool_rows,
                           int32_t n_req, const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                           int32_t max_len, int32_t max_rows_per_req, const int32_t* page_table,
                           int64_t ld_pt, int32_t page_size, int32_t k_blk, int32_t* out_blocks,
                           int32_t* out_pos, int32_t* out_slots, float* scores_out, int64_t ld_scores,
                           void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------
 * IndexShare reuse of a kept selection  ([QSA], section "IndexShare MTP:
 * reusing the QSA selection across draft steps": the QSA selection computed
 * at the draft-extend pass over the tokens the target just accepted is kept
 * for the whole MTP iteration; each draft decode step skips the indexer and
 * reads that frozen selection plus the positions drafted since, so the draft
 * still sees its own in-flight tokens).
 *
 *   cap_blocks [n_cap][k_blk]: kept block ids, e.g. out_blocks of the
 *              draft-extend call (ascending, -1 padded; any order is read
 *              as given, -1 entries skipped).
 *   cap_len    [n_cap]: tokens the kept row saw (its row_len).
 *   cap_row    [n_req]: which kept row serves request r (its last accepted
 *              row).  Rows of request r are the draft rows of this step.
 *   n_extra    drafted columns to reserve, 0 <= n_extra <= 65536 (the MTP
 *              depth N + 1 covers a whole iteration).
 *   out_pos    [n_rows][4*k_blk+3+n_extra] or NULL: token positions.
 *   out_slots  [n_rows][4*k_blk+3+n_extra]: physical KV slots.
 *
 * Row t of request r, seeing L = row_len[t] tokens, with c = cap_row[r] and
 * nb0 = cap_len[c]/4: the positions 4b..4b+3 (those below L) of each kept
 * block b, in the order given, then every position 4*nb0 .. L-1 (the kept
 * row's pending tokens and every token drafted since), then -1.  Device
 * faults: a kept block b >= nb0 is skipped (bit 0); c outside [0, n_cap)
 * gives a row of -1 (bit 0); a list longer than the row is cut at the width
 * (bit 4).  No scores are read and nothing is selected.
 * ------------------------------------------------------------------- */
qsa_status qsa_indexshare_slots(const int32_t* cap_blocks, const int32_t* cap_len, int32_t n_cap,
                                const int32_t* cap_row, int32_t k_blk, int32_t n_extra, int32_t n_req,
                                const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                                const int32_t* page_table, int64_t ld_pt, int32_t page_size,
                                int32_t* out_pos, int32_t* out_slots, void* stream);

/* ---------------------------------------------------------------------
 * Sparse attention over the selected slots  ([QSA]: the compressed keys only
 * index; the final softmax and value aggregation read the original,
 * uncompressed K/V at the selected positions -- sparse GQA over at most
 * 2051 positions.  [SMLA]: the only mask is index >= 0, and a token whose
 * whole selection is masked must not give NaN).
 *
 *   q          [n_rows][h_q][head_dim] BF16 queries (16-byte aligned).
 *   k_cache, v_cache  [n_slots][h_kv][head_dim] BF16: the K and V rows of
 *              every physical KV slot (16-byte aligned).
 *   slots      [n_rows][ld_slots] int32: entries 0 .. n_idx-1 of each row
 *              are read (e.g. out_slots of qsa_indexer_select or
 *              qsa_indexshare_slots); entries < 0 are skipped.
 *   scale      softmax scale (e.g. 1/sqrt(head_dim)).
 *   out        [n_rows][h_q][head_dim] FP32.
 *   lse        [n_rows][h_q] FP32 or NULL: log sum_j exp(scale <q_h, k_j>).
 *   workspace  qsa_sparse_attn_workspace_size(n_rows, h_q, head_dim, n_idx)
 *              bytes (16-byte aligned; 0 bytes when n_idx <= 256).
 *
 * Query head h reads KV head h / (h_q / h_kv).  For each row and query head:
 * out = sum_j softmax_j(scale <q_h, k_j>) v_j over the valid entries, FP32
 * arithmetic on BF16 inputs.  A row with no valid entry gets out = 0 and
 * lse = -inf.  Supported: h_q / h_kv a power of two, up to 16 with
 * head_dim 128, up to 8 with head_dim 256 (else QSA_ERR_UNSUPPORTED).
 * A slot >= n_slots is skipped and latches device fault bit 0.
 * ------------------------------------------------------------------- */
size_t qsa_sparse_attn_workspace_size(int32_t n_rows, int32_t h_q, int32_t head_dim, int32_t n_idx);
qsa_status qsa_sparse_attn(const void* q, const void* k_cache, const void* v_cache, int64_t n_slots,
                           int32_t n_rows, int32_t h_q, int32_t h_kv, int32_t head_dim,
                           const int32_t* slots, int64_t ld_slots, int32_t n_idx, float scale, float* out,
                           float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------
 * Top-k_blk blocks of given block scores, expanded and translated, one
 * call  ([QSA] 512-block selection, 4 token positions per block followed by
 * the pending tokens; [TOPK] selection fused with the page-table transform).
 * The selection half of qsa_indexer_select, for scores that come from
 * elsewhere (qsa_index_scores, or another scorer).
 *
 *   scores     [n_rows][ld_scores] FP32; the candidates of row t are its
 *              entries b < row_len[t]/4.  ld_scores >= max_len/4.
 *   out_blocks [n_rows][k_blk] or NULL: the selected block ids, ascending,
 *              -1 after the first min(k_blk, row_len/4).
 *   out_pos    [n_rows][4*k_blk+3] or NULL: token positions.
 *   out_slots  [n_rows][4*k_blk+3]: physical KV slots, -1 padded.
 * Order and ties as in topk_select.
 * ------------------------------------------------------------------- */
qsa_status qsa_select_blocks(const float* scores, int64_t ld_scores, int32_t n_req,
                             const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                             int32_t max_len, const int32_t* page_table, int64_t ld_pt,
                             int32_t page_size, int32_t k_blk, int32_t* out_blocks, int32_t* out_pos,
                             int32_t* out_slots, void* stream);

/* ---------------------------------------------------------------------
 * The fused decode path: score -> top-k_blk blocks -> expand -> slots, one
 * call  ([QSA] score equation and 512-block selection; [TOPK] selection
 * fused with the page-table transform).
 *
 *   out_blocks [n_rows][k_blk] or NULL: the selected block ids.
 *   out_pos    [n_rows][4*k_blk+3] or NULL: token positions.
 *   out_slots  [n_rows][4*k_blk+3]: physical KV slots, -1 padded.
 *   scores_out [n_rows][ld_scores] or NULL: the FP32 scores the selection
 *              ran on (entries b < row_len/4); when NULL they live in the
 *              workspace.
 * Workspace: when scores_out is NULL the scores live in the workspace, which
 * must hold qsa_indexer_select_workspace_size(n_rows, max_len, k_blk) bytes;
 * when scores_out is given the workspace may be NULL with 0 bytes.  Past the
 * scores (or from its start, with scores_out) a workspace of that size also
 * holds the selection's row plan for contexts of more than 131,072 tokens
 * (see topk_select); without room for it the plan is made on the host.
 * ------------------------------------------------------------------- */
size_t qsa_indexer_select_workspace_size(int32_t n_rows, int32_t max_len, int32_t k_blk);
qsa_status qsa_indexer_select(const void* q, const void* pool, int64_t pool_rows, int32_t n_req,
                              const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                              int32_t max_len, int32_t max_rows_per_req, const int32_t* page_table,
                              int64_t ld_pt, int32_t page_size, int32_t k_blk, int32_t* out_blocks,
                              int32_t* out_pos, int32_t* out_slots, float* scores_out,
                              int64_t ld_scores, void* workspace, size_t workspace_bytes,
                              void* stream);

/* ---------------------------------------------------------------------
 * The fused decode path for callers that cannot allocate device memory.
 * (Library addition with no counterpart in the source pages.)
 *
 * Who needs it: code that must not call cudaMalloc at the point where the
 * indexer runs -- for example an engine whose memory planner hands out every
 * byte up front, a plugin living inside another framework that gives it no
 * allocator, or a latency-critical loop that cannot afford the device-wide
 * synchronisation an allocation may cause.  Such callers cannot size and
 * pass the workspace of qsa_indexer_select, so this
 * call keeps the FP32 scores in a fixed scratch array that is part of the
 * library itself: QSA_NOALLOC_SCRATCH_BYTES bytes of device memory, held on
 * every GPU that loads the library until the process exits.
 *
 * Arguments and results are those of qsa_indexer_select without scores_out
 * and the workspace; the caller still passes (and owns) all inputs and
 * outputs.  The call allocates and frees nothing.
 *
 *  - Limit: n_rows * round_up(max_len/4, 4) * 4 bytes of scores must fit in
 *    QSA_NOALLOC_SCRATCH_BYTES; larger calls return QSA_ERR_UNSUPPORTED and
 *    enqueue nothing.
 *  - Set-up: the first call on each device looks up the scratch array's
 *    device address (cudaGetSymbolAddress) with that device current; make
 *    that first call outside any stream capture.
 *  - Sharing: all calls in the process share the one array per device, and
 *    it keeps whatever the previous call left in it.  Nothing needs to start
 *    at zero (every score the selection reads is written first by the same
 *    call), but two calls whose work overlaps on the GPU -- on different
 *    streams, or from different threads -- race on the array.  Serialise
 *    them (one stream, or events).
 * ------------------------------------------------------------------- */
#define QSA_NOALLOC_SCRATCH_BYTES (16u << 20)
qsa_status qsa_indexer_select_noalloc(const void* q, const void* pool, int64_t pool_rows,
                                      int32_t n_req, const int32_t* req_row_start, int32_t n_rows,
                                      const int32_t* row_len, int32_t max_len,
                                      int32_t max_rows_per_req, const int32_t* page_table,
                                      int64_t ld_pt, int32_t page_size, int32_t k_blk,
                                      int32_t* out_blocks, int32_t* out_pos, int32_t* out_slots,
                                      void* stream);

/* ---------------------------------------------------------------------
 * Prologue tails  (SGLang GLM-5.2 blog, section "Indexer Prologue Fusion":
 * the query path applies RoPE and FP8 quantisation, the key path FP8
 * quantisation before the paged index-cache store; QSA's score has no head
 * gates, so none are applied).
 *
 * qsa_rope_queries: the 4 index heads of row t rotated at position pos[t]
 * (the newest token the row sees, row_len - 1), rotate-half pairs (i, i+64),
 * angle pos * rope_base^(-2i/128), the angle reduced exactly as in
 * qsa_compress_keys; FP32 arithmetic, one rounding to BF16 (nearest even).
 *   q, q_out   [n_rows][4][128] BF16, 16-byte aligned (q_out may equal q).
 *   pos        [n_rows] positions >= 0 (a negative one latches the grouping
 *              fault bit and leaves that row's output unwritten).
 *
 * qsa_quantize_keys_fp8: compressed keys to FP8.  The pages give no layout
 * for FP8 index keys; the one used here: e4m3 codes (1 sign, 4 exponent bits
 * biased by 7, 3 mantissa bits, largest finite 448) with one FP32 scale per
 * key, scale = max_d |k_d| / 448 (FP32 division) and code_d = e4m3(k_d /
 * scale) (FP32 division, nearest value, ties to even, saturating); a zero key
 * gets scale 0 and zero codes.
 *   keys   [n_keys][128] BF16 (16-byte aligned), e.g. a whole pool.
 *   codes  [n_keys][128] bytes (16-byte aligned); scales [n_keys] FP32.
 *
 * qsa_index_scores_fp8 / qsa_indexer_select_fp8: qsa_index_scores and
 * qsa_indexer_select on FP8 keys (codes and scales in place of the BF16
 * pool, same pool-row addressing).  The query is held in FP16 (each BF16
 * element rounded to the nearest binary16 value, exact for magnitudes in
 * [2^-14, 65504)); a key contributes code * scale:
 *   s[t][b] = (1/sqrt(128)) sum_h ReLU( scale_b sum_d f16(q[t][h][d]) code_b[d] ).
 * Up to 4096 requests of up to 8 rows each, on pages holding a multiple of
 * 8 compressed keys (page_size a multiple of 32); other shapes return
 * QSA_ERR_UNSUPPORTED.  Workspace, outputs and errors as for the BF16 calls.
 * ------------------------------------------------------------------- */
qsa_status qsa_rope_queries(const void* q, const int32_t* pos, int32_t n_rows, double rope_base, void* q_out,
                            void* stream);
qsa_status qsa_quantize_keys_fp8(const void* keys, int64_t n_keys, uint8_t* codes, float* scales, void* stream);
qsa_status qsa_index_scores_fp8(const void* q, const uint8_t* codes, const float* scales, int64_t pool_rows,
                                int32_t n_req, const int32_t* req_row_start, int32_t n_rows, const int32_t* row_len,
                                int32_t max_len, int32_t max_rows_per_req, const int32_t* page_table, int64_t ld_pt,
                                int32_t page_size, float* scores, int64_t ld_scores, int64_t n_fill, void* stream);
qsa_status qsa_indexer_select_fp8(const void* q, const uint8_t* codes, const float* scales, int64_t pool_rows,
                                  int32_t n_req, const int32_t* req_row_start, int32_t n_rows,
                                  const int32_t* row_len, int32_t max_len, int32_t max_rows_per_req,
                                  const int32_t* page_table, int64_t ld_pt, int32_t page_size, int32_t k_blk,
                                  int32_t* out_blocks, int32_t* out_pos, int32_t* out_slots, float* scores_out,
                                  int64_t ld_scores, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------
 * Head gates  (SGLang GLM-5.2 blog, section "Indexer Prologue Fusion": the
 * query path scales the index heads by a gate).  QSA's own score has no
 * head weights; with gates g [n_rows][4] (FP32, row-major, 16-byte aligned)
 * every head's rectified dot product is multiplied by its row's gate before
 * the head sum:
 *   s[t][b] = (1/sqrt(128)) sum_h g[t][h] * ReLU(<q[t][h], kbar[b]>).
 * head_gates = NULL is the plain score (qsa_index_scores and
 * qsa_indexer_select are these calls without gates).  Every other argument,
 * the workspace, outputs and errors as for the ungated calls.
 * ------------------------------------------------------------------- */
qsa_status qsa_index_scores_gated(const void* q, const float* head_gates, const void* pool, int64_t pool_rows,
                                  int32_t n_req, const int32_t* req_row_start, int32_t n_rows,
                                  const int32_t* row_len, int32_t max_len, int32_t max_rows_per_req,
                                  const int32_t* page_table, int64_t ld_pt, int32_t page_size, float* scores,
                                  int64_t ld_scores, int64_t n_fill, void* stream);
qsa_status qsa_indexer_select_gated(const void* q, const float* head_gates, const void* pool, int64_t pool_rows,
                                    int32_t n_req, const int32_t* req_row_start, int32_t n_rows,
                                    const int32_t* row_len, int32_t max_len, int32_t max_rows_per_req,
                                    const int32_t* page_table, int64_t ld_pt, int32_t page_size, int32_t k_blk,
                                    int32_t* out_blocks, int32_t* out_pos, int32_t* out_slots, float* scores_out,
                                    int64_t ld_scores, void* workspace, size_t workspace_bytes, void* stream);
/* qsa_decode_step with head gates for the step's query rows (between q and
 * pool; NULL: qsa_decode_step). */
qsa_status qsa_decode_step_gated(const void* new_keys, const int32_t* req_tok_start, const int32_t* req_first_pos,
                                 void* ring, double rope_base, const void* q, const float* head_gates, void* pool,
                                 int64_t pool_rows, int32_t n_req, const int32_t* req_row_start, int32_t n_rows,
                                 const int32_t* row_len, int32_t max_len, int32_t max_rows_per_req,
                                 const int32_t* page_table, int64_t ld_pt, int32_t page_size, int32_t k_blk,
                                 int32_t* out_blocks, int32_t* out_pos, int32_t* out_slots, float* scores_out,
                                 int64_t ld_scores, void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H_ */
