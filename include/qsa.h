/*
 * qsa.h -- C ABI of libqsa.so, the GB300 (sm_103a) QSA token-indexer hot path.
 *
 * The QSA token indexer (pegainfer PR #1160 "score QSA token-indexer blocks in
 * native CUDA" and PR #1178 "select QSA indexer blocks"; metrale layers/qsa.rs)
 * turns a sequence's raw indexer keys and its query rows into a per-row u8
 * visibility mask in three steps:
 *
 *   1. pool   -- each complete 4-token block of raw bf16 keys becomes one block
 *                key: f32 mean -> bf16 -> (1 + w) RMSNorm -> bf16 -> partial
 *                RoPE (first 64 of 128 dims) at the block's first token -> bf16;
 *   2. score  -- S[r, b] = sum_h relu(q_h . k_b) / sqrt(128) over 4 query heads,
 *                each head prepared like a key (norm with q_norm_w, RoPE at the
 *                row's own position);
 *   3. select -- per row at position p: blocks = (p+1)/4, tail = (p+1)%4,
 *                keep = min(budget/4, blocks); the kept blocks are the `keep`
 *                highest scores under the order (score descending, block index
 *                ascending, -0.0 == +0.0); the mask is 1 on their 4 tokens each
 *                and on the tail [4*blocks, p], 0 on every other byte of the row.
 *
 * Fixed geometry: 4 query heads, head dim 128, ratio 4, rotary dim 64.
 *
 * Conventions shared by every entry point
 *  - bf16 values travel as uint16_t bit patterns (the upper half of an f32).
 *  - Pointers marked DEVICE are pointers the GPU can address, owned by the
 *    caller: CUDA device or managed memory, or page-locked host memory (it is
 *    mapped into the unified address space, and the kernels read and write it
 *    in place over the CPU-GPU link, e.g. a decode step's query row, position
 *    and mask row).  Keep the large arrays (block keys, scores) and every
 *    workspace and status word in device memory: atomics and bulk copies
 *    target them.  The library allocates nothing and frees nothing.  `stream`
 *    is a cudaStream_t (NULL = the legacy default stream); every launch is
 *    stream-ordered and asynchronous.
 *  - Arguments are validated on the host before any launch.  A refusal returns
 *    QSA_ERR_INVALID_VALUE and launches nothing.  Refused: negative extents,
 *    NULL pointers with a non-empty extent, pointers or row strides not
 *    16-byte aligned where the comment says so, a budget that is not a positive
 *    multiple of 4 keeping at most 512 blocks, score_cols below tokens/4,
 *    RoPE tables shorter than the positions a call can read, eps < 0 or NaN,
 *    and size products that overflow.
 *  - An empty launch (no rows, no tokens or no blocks) is a no-op returning
 *    QSA_OK.
 *  - Errors that only the device can see (a row position outside [0, tokens),
 *    a visible length outside [0, p+1], a non-finite score inside a
 *    truncating row's block prefix) do not trap: the kernel records the first
 *    one in the caller's status word and leaves that row's output untouched
 *    -- except the mask row of a non-finite score, which the selection may
 *    have partly written before it met the score (the tokens past the row's
 *    complete blocks, or a one-pass selection's bytes; they are then 0 or 1,
 *    and unspecified).  Every other row is complete.
 *    dev_status is a DEVICE int32_t[2] = {code, row}; it must be zero before
 *    the call (qsa_reset_status) and is read with qsa_read_status.
 */
#ifndef QSA_H
#define QSA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QSA_OK = 0,
    QSA_ERR_INVALID_VALUE = 1, /* refused on the host; nothing launched */
    QSA_ERR_LAUNCH = 2,        /* the CUDA runtime refused a launch */
    QSA_ERR_ROW_RANGE = 3,     /* device: pos, visible_len (or key_base) out of range */
    QSA_ERR_NONFINITE = 4,     /* device: NaN/Inf score in a truncating row */
    QSA_ERR_TIMEOUT = 5,       /* device: a bounded wait gave up */
    QSA_ERR_TOKEN_RANGE = 6    /* device: a gathered token or its page lies outside
                                  the page table or the pool */
} qsa_status;

/* Which scorer qsa_score_rows_with runs. */
typedef enum {
    QSA_SCORE_AUTO = 0,    /* host picks: the tile scorer for many rows sharing one key set,
                              else the streaming one */
    QSA_SCORE_SIMT = 1,    /* bandwidth-bound warp-dot scorer (decode shape, any rows) */
    QSA_SCORE_TCGEN05 = 2, /* tcgen05/TMEM/TMA tile scorer; needs key_base == NULL */
    QSA_SCORE_STREAM = 3   /* streaming tcgen05 scorer: each row's 128-block tiles fetched
                              by TMA, scored against its 4 heads (decode shape, any rows) */
} qsa_score_path;

/* Library version (major*10000 + minor*100 + patch). */
int32_t qsa_version(void);

/* Short text for a status code (static storage). */
const char *qsa_status_string(int32_t status);

/*
 * The limit of the bounded device waits a caller may shorten, in SM clock
 * cycles (default 4e9, about 2 s at 2 GHz): the streaming scorers' waits for
 * the block keys they copy into shared memory and for their MMAs
 * (qsa_score_rows on the SIMT and QSA_SCORE_STREAM paths), and the fused
 * decode step's waits for its key copies, its MMAs and its barrier over a
 * row's CTAs (qsa_decode_index_select).  A wait
 * that reaches the limit records QSA_ERR_TIMEOUT with its row in dev_status
 * and the row's output is left unspecified (a fused decode call may then
 * leave its workspace dirty: zero it before the next call); the CTA first
 * lets its own copies and MMAs in flight finish, under the fixed default
 * limit.  Source: PR #1178's review note on
 * environment side effects (a trap left the GPU unusable, so waits report
 * instead of trapping); a short limit lets a test make a wait run out without
 * faulting anything.  The value is process-wide and read when a kernel is
 * launched (a captured CUDA graph keeps the value in force at capture).
 * qsa_set_wait_limit_cycles refuses cycles <= 0 with QSA_ERR_INVALID_VALUE.
 */
qsa_status qsa_set_wait_limit_cycles(int64_t cycles);
int64_t qsa_wait_limit_cycles(void);

/*
 * RoPE cos/sin tables, HOST memory, built on the CPU (no device work).
 * Source: PR #1160 review ("read the cos and sin table that the rope module
 * builds"): the indexer rotates with the same position embeddings as attention,
 * so the tables are inputs of every rotating call.
 * Row p (p < max_pos) of each table is 64 bf16 values [v_0..v_31, v_0..v_31]
 * with v_j = bf16(f32(cos/sin(f32(p * f32(1 / theta^(2j/64)))))).
 * cos_out, sin_out: HOST uint16_t[max_pos * 64], caller-owned.
 * Refuses max_pos < 0, theta <= 0 or non-finite, NULL outputs with max_pos > 0.
 */
qsa_status qsa_rope_tables(int32_t max_pos, double theta, uint16_t *cos_out, uint16_t *sin_out);

/*
 * Pool blocks [first_block, first_block + n_blocks) into block keys.
 * Source: PR #1160 description (block keys: raw keys averaged in float32, cast
 * back to bf16, (1 + w) RMSNorm, partial RoPE at the block's first token);
 * metrale layers/qsa.rs pool_new_blocks (only newly complete blocks).
 *  keys        DEVICE bf16; the raw key of token 4*first_block + t is the 128
 *              values at keys + t*key_stride, t < 4*n_blocks.  16-byte aligned;
 *              key_stride >= 128 and a multiple of 8 (640 reads a fused q|k
 *              row buffer offset to column 512; 128 reads a compact key cache).
 *  k_norm_w    DEVICE bf16[128], 16-byte aligned; the norm weight is 1 + w.
 *  cos_t/sin_t DEVICE bf16[table_rows * 64] from qsa_rope_tables, 16-byte
 *              aligned; table_rows must exceed 4*(first_block + n_blocks - 1).
 *  eps         RMSNorm epsilon (>= 0).
 *  block_keys  DEVICE bf16 key cache; block b is written to block_keys + b*128.
 *              16-byte aligned.  Nothing else is written.
 */
qsa_status qsa_pool_blocks(const uint16_t *keys, int64_t key_stride, int32_t first_block,
                           int32_t n_blocks, const uint16_t *k_norm_w, const uint16_t *cos_t,
                           const uint16_t *sin_t, int32_t table_rows, float eps,
                           uint16_t *block_keys, void *stream);

/*
 * Score query rows against block keys.
 * Source: PR #1160 description (sum_h relu(q_h . k_b) / sqrt(indexer_head_dim),
 * relu per head before the head sum, written as a comparison so a NaN stays
 * NaN; rows/visible_len as separate device arrays; only the visible prefix of
 * each score row is written, the rest is left untouched).
 *  q           DEVICE bf16; row i's four query heads are the 512 values at
 *              q + i*q_stride (q_stride >= 512, multiple of 8; 640 for a fused
 *              q|k buffer).  16-byte aligned.
 *  pos         DEVICE int32[n_rows]: row i's position p (0 <= p < tokens).
 *  visible_len DEVICE int32[n_rows] or NULL (= p + 1): the row sees its first
 *              visible_len tokens, so blocks = visible_len / 4.
 *  tokens      positions are < tokens.
 *  q_norm_w    DEVICE bf16[128] query norm weight (used as 1 + w).
 *  cos_t/sin_t DEVICE RoPE tables with table_rows >= tokens.
 *  block_keys  DEVICE bf16 pooled keys; row i reads block b at
 *              block_keys + (key_base[i] + b)*128.  16-byte aligned.  With
 *              key_base == NULL the buffer must be readable for tokens/4
 *              blocks (the tensor-core scorer fetches whole 128-block tiles;
 *              blocks past a row's prefix are read but never used).
 *  key_base    DEVICE int64[n_rows] or NULL (= 0): per-row block offset, so one
 *              call can score rows of different sequences.  Only a row's own
 *              blocks are read.  The streaming tcgen05 scorer addresses
 *              blocks below 2^31 (512 GiB of keys): a row whose key_base +
 *              blocks passes that, or a negative key_base, is recorded as
 *              QSA_ERR_ROW_RANGE.
 *  scores      DEVICE f32, row stride score_cols (>= tokens/4, multiple of 4;
 *              spare capacity allowed), 16-byte aligned.  Row i gets entries
 *              b < blocks; entries past that are not written.
 *  dev_status  DEVICE int32[2] status word (see above).
 *  workspace   DEVICE scratch owned by the caller, or NULL; 16-byte aligned.
 *              The tensor-core scorer needs qsa_score_workspace_bytes(n_rows)
 *              bytes for the prepared query heads; its contents on entry do
 *              not matter and are overwritten.  The streaming scorers use
 *              none.
 * qsa_score_rows picks the scorer itself (QSA_SCORE_AUTO): the tensor-core
 * tile scorer for 64 or more rows sharing one key set (key_base == NULL) when
 * the workspace is large enough, the streaming tcgen05 scorer otherwise (its
 * scores equal the fused decode launch's: the same MMA per block).
 */
qsa_status qsa_score_rows(const uint16_t *q, int64_t q_stride, const int32_t *pos,
                          const int32_t *visible_len, int32_t n_rows, int32_t tokens,
                          const uint16_t *q_norm_w, const uint16_t *cos_t, const uint16_t *sin_t,
                          int32_t table_rows, float eps, const uint16_t *block_keys,
                          const int64_t *key_base, float *scores, int64_t score_cols,
                          int32_t *dev_status, void *workspace, int64_t workspace_bytes,
                          void *stream);

/* Workspace bytes the tensor-core scorer needs for n_rows query rows
 * (1024 per row: 4 prepared heads x 128 bf16); -1 for n_rows < 0. */
int64_t qsa_score_workspace_bytes(int32_t n_rows);

/* qsa_score_rows with an explicit scorer; QSA_SCORE_TCGEN05 refuses key_base != NULL
 * and a workspace smaller than qsa_score_workspace_bytes(n_rows); QSA_SCORE_SIMT and
 * QSA_SCORE_STREAM take any rows and no workspace.  The three give the same scores
 * within the scoring tolerance; the two tcgen05 scorers give identical ones. */
qsa_status qsa_score_rows_with(const uint16_t *q, int64_t q_stride, const int32_t *pos,
                               const int32_t *visible_len, int32_t n_rows, int32_t tokens,
                               const uint16_t *q_norm_w, const uint16_t *cos_t,
                               const uint16_t *sin_t, int32_t table_rows, float eps,
                               const uint16_t *block_keys, const int64_t *key_base,
                               float *scores, int64_t score_cols, int32_t *dev_status,
                               int32_t path, void *workspace, int64_t workspace_bytes,
                               void *stream);

/*
 * qsa_score_rows_noalloc -- the tensor-core scorer without a caller workspace.
 * The pages have no counterpart to this entry point.  It serves callers that
 * cannot allocate device memory when they score: engines that reserve all free
 * HBM up front (for their KV cache) and forbid allocation afterwards, code
 * running where the CUDA allocator may not be called (a host callback), and
 * real-time loops that cannot take an allocation's latency or failure
 * mid-step.  Arguments are those of qsa_score_rows with key_base == NULL and
 * no workspace; the library allocates nothing here either: the query-prep
 * workspace is a file-scope device array of QSA_NOALLOC_MAX_ROWS * 1024 bytes
 * (8 MiB) that every GPU loading the library holds until exit.
 *  - n_rows > QSA_NOALLOC_MAX_ROWS is refused with QSA_ERR_INVALID_VALUE before
 *    any launch; other refusals are qsa_score_rows_with's (QSA_SCORE_TCGEN05).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; QSA_ERR_LAUNCH if the
 *    lookup fails.  Make the first call on each device before any stream
 *    capture.  After a device reset (cudaDeviceReset, or the primary context
 *    released and created again) the next call sees a new context ID and
 *    looks the address up again; make that call before any capture too.
 *  - Every call shares the one array and it keeps the last call's contents;
 *    each call overwrites all of it that it reads, so nothing must start at
 *    zero.  Calls that overlap on the GPU (unordered streams or host threads
 *    on one device) race on it: order them.
 */
#define QSA_NOALLOC_MAX_ROWS 8192
qsa_status qsa_score_rows_noalloc(const uint16_t *q, int64_t q_stride, const int32_t *pos,
                                  const int32_t *visible_len, int32_t n_rows, int32_t tokens,
                                  const uint16_t *q_norm_w, const uint16_t *cos_t,
                                  const uint16_t *sin_t, int32_t table_rows, float eps,
                                  const uint16_t *block_keys, float *scores, int64_t score_cols,
                                  int32_t *dev_status, void *stream);

/*
 * Exact top-(budget/4) block selection into a u8 visibility mask.
 * Source: PR #1178 "Exact semantics" (blocks, tail, keep; canonical order
 * descending score then ascending block index; threshold-equal blocks fill the
 * remaining slots in block order; -0.0 ties +0.0; the tail is always visible;
 * a row with blocks <= budget/4 writes its whole visible prefix; a non-finite
 * score in a truncating row's prefix is an error; explicit score_cols).
 *  scores      DEVICE f32, row i at scores + i*score_cols, 16-byte aligned,
 *              score_cols >= tokens/4 and a multiple of 4.  Only entries
 *              b < (pos[i]+1)/4 are read, and none for rows under the budget.
 *  pos         DEVICE int32[n_rows].
 *  budget      positive multiple of 4, budget/4 <= 512.
 *  mask        DEVICE u8[n_rows * tokens]; row i at mask + i*tokens (any
 *              alignment).  Every byte of a valid row is written.
 */
qsa_status qsa_select_mask(const float *scores, int64_t score_cols, const int32_t *pos,
                           int32_t n_rows, int32_t tokens, int32_t budget, uint8_t *mask,
                           int32_t *dev_status, void *stream);

/*
 * The whole hot path on one stream: pool the newly complete blocks, score the
 * rows, select.  Source: metrale layers/qsa.rs decode_select (ingest -> pool
 * new blocks -> prepare q -> score -> top-k -> expand with the tail), with the
 * host sort replaced by the on-device selection of PR #1178.
 *  keys, key_stride, pool_first_block, pool_n_blocks, k_norm_w: as
 *              qsa_pool_blocks (pool_n_blocks == 0 pools nothing);
 *  q, q_stride, pos, n_rows, tokens, q_norm_w: as qsa_score_rows (every row
 *              sees p + 1 tokens and reads block_keys from offset 0);
 *  cos_t, sin_t, table_rows, eps: shared by pool and score;
 *  budget, mask: as qsa_select_mask;
 *  block_keys  DEVICE pooled-key cache (read and written);
 *  scores      DEVICE f32 work buffer of n_rows * score_cols (its contents
 *              afterwards are the rows' scores);
 *  workspace, workspace_bytes: as qsa_score_rows (NULL selects the streaming
 *              scorer).
 */
qsa_status qsa_index_select(const uint16_t *keys, int64_t key_stride, int32_t pool_first_block,
                            int32_t pool_n_blocks, const uint16_t *k_norm_w, const uint16_t *q,
                            int64_t q_stride, const int32_t *pos, int32_t n_rows, int32_t tokens,
                            const uint16_t *q_norm_w, const uint16_t *cos_t,
                            const uint16_t *sin_t, int32_t table_rows, float eps, int32_t budget,
                            uint16_t *block_keys, float *scores, int64_t score_cols,
                            uint8_t *mask, int32_t *dev_status, void *workspace,
                            int64_t workspace_bytes, void *stream);

/*
 * Bytes of the workspace qsa_decode_index_select needs: per row, a 65536-bin
 * histogram, a few counters and room for tokens/4 candidates.  -1 for
 * negative arguments.
 */
int64_t qsa_decode_workspace_bytes(int32_t n_rows, int32_t tokens);

/*
 * The same operation as qsa_index_select (pool the newly complete blocks,
 * score every row, select), for decode-sized row counts, as ONE cooperative
 * launch: each CTA copies a 128-block tile of a row's keys with TMA and
 * scores it on the tensor cores (the CTAs whose ranges hold new blocks pool
 * them while the tile lands), the row's CTAs build its histogram, meet at a
 * bounded grid barrier, find the bin of the keep-th key, write their own
 * blocks' mask bytes and list that bin's keys; the row's last CTA clears the
 * workspace and resolves the listed keys.  (New blocks at or past tokens/4
 * are pooled by a separate launch first.)  Source: metrale layers/qsa.rs
 * decode_select (score then top-k each decode step), PR #1160 (scores),
 * PR #1178 "Exact semantics" (selection).
 * The scores equal those of qsa_index_select's tensor-core scorer (same MMA
 * shape and accumulation order) and the mask is the selector's on them.
 * When the rows' CTAs cannot all be resident at once, the call falls back to
 * the streaming tcgen05 scorer and the selector as two launches (the
 * workspace is not used; the same scores, since that scorer runs the same
 * MMA per block, and the same mask).
 *  arguments   as qsa_index_select, except:
 *  decode_ws   DEVICE workspace of at least qsa_decode_workspace_bytes(n_rows,
 *              tokens) bytes, 16-byte aligned, ZERO before the first call.
 *              Each call that completes leaves it zero again; after a call
 *              that reported an error on the device it may be left dirty and
 *              must be zeroed before the next call.  Calls sharing one
 *              workspace must be stream-ordered.
 *  Returns QSA_ERR_INVALID_VALUE for a missing, small or unaligned workspace
 *  (rows and tokens non-zero), or any argument qsa_index_select refuses.
 */
qsa_status qsa_decode_index_select(const uint16_t *keys, int64_t key_stride,
                                   int32_t pool_first_block, int32_t pool_n_blocks,
                                   const uint16_t *k_norm_w, const uint16_t *q, int64_t q_stride,
                                   const int32_t *pos, int32_t n_rows, int32_t tokens,
                                   const uint16_t *q_norm_w, const uint16_t *cos_t,
                                   const uint16_t *sin_t, int32_t table_rows, float eps,
                                   int32_t budget, uint16_t *block_keys, float *scores,
                                   int64_t score_cols, uint8_t *mask, int32_t *dev_status,
                                   void *decode_ws, int64_t decode_ws_bytes, void *stream);

/*
 * The selected token list of each mask row: the tokens t < tokens whose mask
 * byte is non-zero, ascending.  Source: metrale layers/qsa.rs decode_select,
 * after its top-k (every kept block's four tokens, blocks ascending, then the
 * tail -- exactly the set bytes of the mask qsa_select_mask writes).
 *  mask     DEVICE u8 [n_rows * tokens], row i at mask + i*tokens (any alignment).
 *  sel      DEVICE int32, row i at sel + i*sel_cols; the first
 *           min(count, sel_cols) tokens are written, the rest of the row is
 *           left alone.  For a selection mask, budget + 3 columns always suffice.
 *  n_sel    DEVICE int32 [n_rows]: each row's count of set bytes (a count above
 *           sel_cols means the list was cut).
 */
qsa_status qsa_mask_tokens(const uint8_t *mask, int32_t n_rows, int32_t tokens, int32_t *sel,
                           int64_t sel_cols, int32_t *n_sel, void *stream);

/*
 * Gather the K and V rows of each row's selected tokens from a paged cache into
 * a contiguous scratch.  Source: metrale layers/qsa.rs decode_select and its
 * QsaSelection (a contiguous NHD k/v scratch that the paged decode attention
 * reads through an identity block table).
 *  k_pool, v_pool  DEVICE bf16 [pool_pages * page_size, width], 16-byte aligned;
 *           width = kv_heads * head_dim values per token, a multiple of 8.
 *  table    DEVICE int32: row i's page table at table + i*table_cols
 *           (table_cols = 0: one table shared by every row), table_len entries;
 *           token t of the row is in physical page table[t / page_size], slot
 *           t % page_size.
 *  sel, sel_cols, n_sel: as qsa_mask_tokens writes them; row i gathers its
 *           first min(n_sel[i], max_sel) tokens (max_sel <= sel_cols, out_rows).
 *  k_out, v_out  DEVICE bf16 [n_rows * out_rows, width], 16-byte aligned: row i's
 *           j-th token at (i*out_rows + j).
 *  A token outside [0, table_len * page_size), or a table entry outside
 *  [0, pool_pages), is recorded as QSA_ERR_TOKEN_RANGE and not read.
 */
qsa_status qsa_gather_kv(const uint16_t *k_pool, const uint16_t *v_pool, int32_t width,
                         int32_t pool_pages, const int32_t *table, int32_t table_len,
                         int64_t table_cols, int32_t page_size, const int32_t *sel,
                         int64_t sel_cols, const int32_t *n_sel, int32_t n_rows, int32_t max_sel,
                         uint16_t *k_out, uint16_t *v_out, int64_t out_rows, int32_t *dev_status,
                         void *stream);

/*
 * Attention of each query row over its selected tokens only.  Source: atlas
 * layers/qsa_select.rs prefill_select (a row past the inert bound gets its
 * attention context replaced by attention over exactly its selected set --
 * kept blocks' tokens and the tail -- read from the paged K/V cache through
 * the sequence's block table, nq query heads over nkv KV heads, a 1/sqrt(d)
 * scale); metrale layers/qsa.rs module comment (the top budget/ratio blocks
 * plus the incomplete tail).
 *  q        DEVICE bf16, row i at q + i*q_stride: nq heads of head_dim values
 *           (already rotated), 16-byte aligned, q_stride a multiple of 8 and
 *           >= nq*head_dim.  Query head h reads KV head h / (nq / nkv).
 *  k_pool, v_pool  DEVICE bf16 [pool_pages * page_size, nkv, head_dim],
 *           16-byte aligned; head_dim is 128 or 256.
 *  table, table_len, table_cols, page_size: as in qsa_gather_kv (token t of
 *           row i is in page table[i*table_cols + t / page_size], slot
 *           t % page_size; table_cols = 0 shares one table).
 *  sel, sel_cols, n_sel: the selected tokens as qsa_mask_tokens writes them;
 *           row i attends its first min(n_sel[i], max_sel) tokens
 *           (max_sel <= sel_cols).  A row with none gets zeros.
 *  scale    multiplies every logit q_h . k (finite; typically 1/sqrt(head_dim)).
 *  out      DEVICE bf16, row i at out + i*out_stride (nq*head_dim values),
 *           16-byte aligned, out_stride a multiple of 8 and >= nq*head_dim.
 *  Softmax and accumulation run in f32 with the weights rounded to bf16 for
 *  the weighted sum of V (its normaliser uses the same rounded weights).  A
 *  token outside the table, or a table entry outside the pool, is recorded
 *  as QSA_ERR_TOKEN_RANGE and left out; a row that reports it has an
 *  unspecified output.
 */
qsa_status qsa_sparse_attn(const uint16_t *q, int64_t q_stride, int32_t nq, int32_t nkv,
                           int32_t head_dim, const uint16_t *k_pool, const uint16_t *v_pool,
                           int32_t pool_pages, int32_t page_size, const int32_t *table,
                           int32_t table_len, int64_t table_cols, const int32_t *sel,
                           int64_t sel_cols, const int32_t *n_sel, int32_t n_rows, int32_t max_sel,
                           float scale, uint16_t *out, int64_t out_stride, int32_t *dev_status,
                           void *stream);

/*
 * The indexer's qk projection of normed hidden states: y = x W^T in bf16 with
 * f32 accumulation, rounded once to bf16.  Source: atlas layers/qsa_select.rs
 * prefill_select (each 2048-row slab of the normed hidden states is projected
 * hidden -> 640, the fused q|k row that q-prep, pooling and scoring read).
 *  x        DEVICE bf16 [n_rows, hidden], row stride x_stride (a multiple of 8,
 *           >= hidden), 16-byte aligned; hidden a positive multiple of 8.
 *  w        DEVICE bf16 [out_cols, hidden] (a linear layer's [out, in]
 *           weight), contiguous, 16-byte aligned; out_cols a multiple of 16.
 *  y        DEVICE bf16 [n_rows, out_cols], row stride y_stride (a multiple
 *           of 8, >= out_cols), 16-byte aligned.
 *  n_rows <= 65535 * 128.  A bounded wait that gives up is QSA_ERR_TIMEOUT.
 */
qsa_status qsa_qk_proj(const uint16_t *x, int64_t x_stride, const uint16_t *w, int32_t n_rows,
                       int32_t hidden, int32_t out_cols, uint16_t *y, int64_t y_stride,
                       int32_t *dev_status, void *stream);

/* Zero a DEVICE status word (stream-ordered). */
qsa_status qsa_reset_status(int32_t *dev_status, void *stream);

/* Copy a DEVICE status word to the host; synchronises `stream` first. */
qsa_status qsa_read_status(const int32_t *dev_status, void *stream, int32_t *host_code,
                           int32_t *host_row);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
