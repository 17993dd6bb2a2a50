/*
 * bsa_topk.h -- C ABI of the GB300 (sm_103a) block-sparse attention top-k
 * selection library.
 *
 * The operations follow the buffer contracts of the vLLM MiniMax-M3 indexer
 * as described in these PR reports:
 *   [47502] "[Minimax-M3] Using tok_sparse_select from MSA instead of triton
 *           kernels" -- one unified token-major score buffer
 *           [total_q, H, max_k_tiles], rows bounded by the causal page count
 *           cdiv(seq_pos + 1, 128), init/local blocks force-included, the
 *           unwritten tail pre-filled with -inf, a token-major [T, H, topk]
 *           int32 output (sections 实现拆解 items 2-4 and 关键源码片段,
 *           indexer_msa.py).
 *   [55235] "[ROCm][Perf] Tune MiniMax-M3 decode top-k for short contexts" --
 *           a launch policy keyed on the block capacity with explicit 128/129
 *           boundaries, a split selector with an adaptive final merge whose
 *           counters survive CUDA-graph replay, and a total order covering
 *           NaN, +-Inf, +-0 and ties (sections 执行摘要, 实现拆解, 评论区精华).
 *   [47984] "[ROCm][MiniMax-M3][Spec Decode] Support speculative decode with
 *           AITER sparse PA" -- speculative-decode rows row = req*dql +
 *           local_q, query position seq_len[req] - dql + local_q, page-16
 *           sparse block-table rows with a per-row sparse context length,
 *           padded rows (seq_len 0) giving an empty context, and a hardened
 *           validity mask (sections 实现拆解 items 1-3, 关键源码片段).
 *
 * Conventions for every call:
 *  - Pointers named in the signature are DEVICE pointers owned by the caller
 *    (except where a parameter says "host"); the library allocates nothing.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous on that stream.  Every call except
 *    bsa_topk_select_noalloc (see its own note) can be captured in a CUDA
 *    graph.
 *  - Outputs are written in full; callers need not clear them first.
 *  - Return value: BSA_OK (0) on success; a negative BSA_ERR_* when the host
 *    rejects the arguments (nothing is launched); a positive cudaError_t when
 *    a launch fails.
 *
 * Total order of scores (reading of [55235]): IEEE 754-2019 clause 5.10
 * totalOrder on the raw bits: -NaN < -Inf < negative < -0 < +0 < positive <
 * +Inf < +NaN, NaNs ordered by payload away from zero.  Equal bit patterns
 * go to the lower block id.
 */
#ifndef BSA_TOPK_H_
#define BSA_TOPK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define BSA_OK 0
#define BSA_ERR_NULL (-1)      /* a required pointer is NULL                   */
#define BSA_ERR_SHAPE (-2)     /* a size is negative, zero where it must not be, or too large */
#define BSA_ERR_TOPK (-3)      /* K < 1, K > BSA_MAX_TOPK, K > M, or K < num_init + num_local */
#define BSA_ERR_DTYPE (-4)     /* unknown score dtype                           */
#define BSA_ERR_WORKSPACE (-5) /* workspace missing, too small or misaligned    */
#define BSA_ERR_ROWS (-6)      /* T != num_reqs * decode_query_len              */
#define BSA_ERR_ALIGN (-7)     /* scores pointer not aligned to its element size */
#define BSA_ERR_CAPACITY (-8)  /* request needs more than the built-in scratch  */

/* ---- constants ---------------------------------------------------------- */
#define BSA_PAGE_SIZE 128              /* tokens per sparse block ([47502] PAGE_SIZE) */
#define BSA_SUB_PAGE_SIZE 16           /* tokens per sparse-table entry ([47984] page-16) */
#define BSA_PAGES_PER_SPARSE_BLOCK 8   /* 128 / 16 */
#define BSA_MAX_TOPK 1024
#define BSA_MAX_K_TILES 65536          /* block ids must fit 16 bits */

/* score element types */
#define BSA_DTYPE_BF16 0
#define BSA_DTYPE_FP32 1

/* selector paths chosen by the launch policy */
#define BSA_PATH_ROW 0      /* one warp streams a whole row                 */
#define BSA_PATH_SPLIT 1    /* several warps per row + last-arriver merge   */
#define BSA_PATH_GROUP 2    /* 4 lanes per row, 8 rows per warp (K <= 32)   */
#define BSA_PATH_PAIR 3     /* 2 lanes per row, 16 rows per warp (K <= 32)  */
#define BSA_PATH_OCTET 4    /* 8 lanes per row, 4 rows per warp (K <= 64)   */
#define BSA_PATH_WIDE 5     /* 32 lanes per row, bf16 rows > 2 KB (K <= 64) */

typedef struct bsa_launch_policy {
    int32_t path;             /* BSA_PATH_*                                   */
    int32_t vecs_per_lane;    /* 16-byte vectors each lane holds per pass     */
    int32_t chunks_per_row;   /* warps cooperating on one row (1 = no split)  */
    int32_t reps_per_lane;    /* threshold-estimate representatives per lane */
    int32_t warps_per_cta;
    int32_t grid;             /* CTAs launched                                */
    int32_t cand_capacity;    /* candidate buffer entries per warp            */
    int32_t smem_bytes;       /* dynamic shared memory per CTA                */
    int32_t long_rows;        /* 1: rows whose range exceeds 2 KB are left to a
                                 second, wide-path launch over a list of them */
    int32_t long_grid;        /* CTAs of that launch (0 when long_rows is 0)  */
} bsa_launch_policy_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* bsa_status_string(int status);

/* Causal page count of decode rows ([47502] 关键源码片段, indexer_msa.py
 * metadata: the number of 128-token pages that cover positions 0 .. pos;
 * row mapping of [47984]):
 *   row = req * decode_query_len + local_q,
 *   pos = seq_lens[req] - decode_query_len + local_q,
 *   num_valid_pages[row] = pos >= 0 ? cdiv(pos + 1, 128) : 0.
 * seq_lens: int32[num_reqs]; num_valid_pages: int32[num_reqs * decode_query_len].
 * Errors: BSA_ERR_NULL, BSA_ERR_SHAPE (num_reqs < 0 or decode_query_len < 1). */
int bsa_num_valid_pages_decode(const int32_t* seq_lens, int64_t num_reqs,
                               int32_t decode_query_len, int32_t* num_valid_pages,
                               void* stream);

/* Causal page count of varlen rows ([47502] "batch-wide inputs for
 * sparse_topk_select": topk_cu_seqlens_q, topk_prefix_lens): sequence i owns
 * rows [cu_seqlens_q[i], cu_seqlens_q[i+1]) and its j-th query token sits at
 * position prefix_lens[i] + j.  Rows in [0, total_q) that no sequence owns
 * get 0.  cu_seqlens_q: int32[num_seqs + 1], non-decreasing;
 * prefix_lens: int32[num_seqs]; num_valid_pages: int32[total_q].
 * Errors: BSA_ERR_NULL, BSA_ERR_SHAPE. */
int bsa_num_valid_pages_varlen(const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                               int64_t num_seqs, int64_t total_q, int32_t* num_valid_pages,
                               void* stream);

/* Bytes of device workspace bsa_topk_select / bsa_topk_select_sparse_table
 * need for these sizes on the current device (0 when the launch policy keeps
 * every row in one warp and leaves none to a second launch).  The workspace
 * holds the per-chunk candidate lists and the merge tickets of the split
 * path, or the list of rows longer than 2 KB and its counter (long_rows in
 * the policy).  Host-only; launches nothing. */
size_t bsa_topk_workspace_bytes(int64_t T, int64_t H, int64_t M, int32_t K, int32_t dtype);

/* Batched causal top-k over the unified token-major score buffer
 * ([47502] sparse_topk_select contract).
 *   scores: element (t, h, b) at scores[t*token_stride + h*head_stride + b],
 *           dtype BSA_DTYPE_BF16 or BSA_DTYPE_FP32, for b < M; only the
 *           causal prefix b < v_t = min(M, num_valid_pages[t]) is read, so
 *           the tail may hold anything (the pages fill it with -inf) and M
 *           may be the capture-time capacity.
 *   num_valid_pages: int32[T].
 *   Row (t, h) selects n = min(K, v_t) block ids: the init blocks
 *   [0, min(num_init, v_t)), the local blocks [max(v_t - num_local, 0), v_t),
 *   and the best remaining ids by (totalOrder of the score descending, id
 *   ascending).  out_idx: int32, row (t, h) at out_idx + t * out_token_stride
 *   + h * out_head_stride with its K slots contiguous; slots [0, n) hold the
 *   selected ids in ascending order, slots [n, K) hold -1.  The token-major
 *   [T, H, K] buffer of [47502] (实现拆解 item 4) has strides (H*K, K); a
 *   head-major [H, T, K] buffer, the layout the Triton consumers of the
 *   vLLM PR #49149 report keep (实现拆解 items 1-2, transpose(0, 1)), has
 *   (K, T*K).  Layouts in which two rows could overlap are rejected
 *   (BSA_ERR_SHAPE).
 *   workspace: device memory of at least bsa_topk_workspace_bytes(...) bytes,
 *   256-byte aligned, any contents.  When it is needed the call first clears
 *   the merge tickets with one cudaMemsetAsync on `stream` (captured as a
 *   memset node in a CUDA graph, so replays start from zero too); the merging
 *   warp also sets its ticket back to 0.  May be NULL when the required size
 *   is 0.  Calls that share a workspace must not overlap on the GPU.
 * Errors: BSA_ERR_NULL, BSA_ERR_SHAPE (T, H < 0; M < 1 or > BSA_MAX_K_TILES;
 * strides too small), BSA_ERR_TOPK, BSA_ERR_DTYPE, BSA_ERR_ALIGN,
 * BSA_ERR_WORKSPACE. */
int bsa_topk_select(const void* scores, int32_t dtype, int64_t T, int64_t H, int64_t M,
                    int64_t token_stride, int64_t head_stride, const int32_t* num_valid_pages,
                    int32_t K, int32_t num_init, int32_t num_local, int32_t* out_idx,
                    int64_t out_token_stride, int64_t out_head_stride, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Page-16 sparse block table ([47984] minimax_m3_build_sparse_block_table_decode
 * and the hardened _build_sparse_block_table kernels).
 *   topk_idx: int32[T, H, K], any ids; T must equal num_reqs * decode_query_len.
 *   Row (t, h): req = t / dql, local_q = t % dql,
 *   causal_len = max(seq_lens[req] - dql + local_q + 1, 0).  The ids b with
 *   0 <= b < min(cdiv(causal_len, 128), max_blocks) are kept once each and
 *   sorted ascending; the j-th kept block fills entries [8j, 8j + 8) with
 *   block_table[req * max_blocks + b] * 8 + p for the pages p whose first
 *   token b*128 + 16p lies before causal_len, and 0 otherwise.  All other
 *   entries are 0.  sparse_ctx = sum over kept blocks of
 *   min(128, causal_len - 128 b).  Padded rows (seq_len 0) give ctx 0 and an
 *   all-zero row.
 *   block_table: int32[num_reqs, max_blocks]; seq_lens: int32[num_reqs];
 *   sparse_bt: int32[T, H, K * 8]; sparse_ctx: int32[T, H].
 * Errors: BSA_ERR_NULL, BSA_ERR_SHAPE, BSA_ERR_TOPK (K < 1 or > BSA_MAX_TOPK),
 * BSA_ERR_ROWS (the page's assert total_q == batch * decode_query_len). */
int bsa_build_sparse_block_table(const int32_t* topk_idx, int64_t T, int64_t H, int32_t K,
                                 const int32_t* block_table, int64_t num_reqs,
                                 int64_t max_blocks, const int32_t* seq_lens,
                                 int32_t decode_query_len, int32_t* sparse_bt,
                                 int32_t* sparse_ctx, void* stream);

/* Fused decode selector with the sparse-table epilogue ([55235]
 * EMIT_SPARSE_TABLE; [47984] row mapping): for T = num_reqs * dql decode
 * rows, computes the causal page count from seq_lens, runs the selection of
 * bsa_topk_select, and writes the sparse table of
 * bsa_build_sparse_block_table for the selected ids without a round trip of
 * the ids through memory.  out_idx may be NULL (ids not wanted); when given, its
 * layout follows out_token_stride / out_head_stride as for bsa_topk_select
 * (the sparse table and ctx are always token-major).  Results are
 * identical to bsa_num_valid_pages_decode + bsa_topk_select +
 * bsa_build_sparse_block_table.  Workspace rules as for bsa_topk_select
 * (size from bsa_topk_workspace_bytes(T, H, M, K, dtype)).
 * Errors: as bsa_topk_select and bsa_build_sparse_block_table. */
int bsa_topk_select_sparse_table(const void* scores, int32_t dtype, int64_t num_reqs,
                                 int32_t decode_query_len, int64_t H, int64_t M,
                                 int64_t token_stride, int64_t head_stride,
                                 const int32_t* seq_lens, int32_t K, int32_t num_init,
                                 int32_t num_local, const int32_t* block_table,
                                 int64_t max_blocks, int32_t* out_idx,
                                 int64_t out_token_stride, int64_t out_head_stride,
                                 int32_t* sparse_bt, int32_t* sparse_ctx, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Limits of the fused index score + select. */
#define BSA_MAX_INDEX_DIM 1024       /* index head dimension D                    */
#define BSA_MAX_INDEX_QUERIES 16     /* decode_query_len * H query rows per request */

/* Fused index score + select (+ optional sparse table) of decode rows
 * ([47502] 实现拆解 items 1-3: the decode score kernel writes score_out =
 * unified_scores[:nd] and one top-k pass selects from it; here both run in
 * one launch).  The pages do not print the score formula.  Reading taken:
 * one pooled bf16 index key per physical 128-token block (page = sparse block
 * = index-K block, [47502] 关键源码片段), shared by the index heads, and
 *   score[t, h, b] = sum_d q_idx[t, h, d] * k_idx[block_table[req, b], d]
 * accumulated in fp32 with no scale factor (item 6 removed sm_scale), for
 * the causal blocks b < v_t = min(M, cdiv(pos + 1, 128)) of each decode row
 * (t = req * decode_query_len + local_q, pos = seq_lens[req] -
 * decode_query_len + local_q).  A causal block with no usable key (b >=
 * max_blocks, or a physical id outside [0, num_phys_blocks)) scores -inf.
 *   q_idx: bf16 [T, H, D], 16-byte aligned; k_idx: bf16 [num_phys_blocks, D],
 *   16-byte aligned; D a multiple of 8, at most BSA_MAX_INDEX_DIM;
 *   decode_query_len * H at most BSA_MAX_INDEX_QUERIES.
 *   scores: fp32 unified buffer, element (t, h, b) at t * token_stride +
 *   h * head_stride + b; the causal entries b < v_t are written, the rest is
 *   left as it is (the pages pre-fill it with -inf).
 *   The selection over the written scores is that of
 *   bsa_topk_select_sparse_table (same K, num_init, num_local, output
 *   layouts); sparse_bt / sparse_ctx may both be NULL (no table).
 *   Needs no workspace.
 * Errors: BSA_ERR_NULL, BSA_ERR_SHAPE, BSA_ERR_TOPK, BSA_ERR_ALIGN. */
int bsa_index_score_topk_select(const void* q_idx, const void* k_idx, int64_t num_phys_blocks,
                                int64_t H, int64_t D, const int32_t* block_table,
                                int64_t max_blocks, const int32_t* seq_lens, int64_t num_reqs,
                                int32_t decode_query_len, float* scores, int64_t M,
                                int64_t token_stride, int64_t head_stride, int32_t K,
                                int32_t num_init, int32_t num_local, int32_t* out_idx,
                                int64_t out_token_stride, int64_t out_head_stride,
                                int32_t* sparse_bt, int32_t* sparse_ctx, void* stream);

/* Largest number of query heads sharing one KV head in the attention call. */
#define BSA_MAX_ATTN_GROUP 8

/* Sparse decode attention over the page-16 sparse block table: the consumer
 * of bsa_topk_select_sparse_table's output ([47984] 实现拆解 items 1-2, the
 * decode sparse paged attention reading the page-16 table and its sparse
 * context length; [47502] 实现拆解 item 5).  The pages show the interface
 * only.  Readings taken: index head h selects for KV head h, shared by G
 * query heads; the KV cache is paged in 16-token pages; row (t, h) attends to
 * its first ctx = sparse_ctx[t, h] table tokens, token j in page
 * sparse_bt[t, h, j / 16] at slot j % 16; and
 *   out[t, h, g] = sum_j softmax_j(scale * q[t, h, g] . k_j) v_j
 * with fp32 arithmetic.  A row with an empty context yields zeros; a token
 * whose page id lies outside [0, num_pages) takes no part.
 *   q: bf16 [T, H, G, D]; k_cache, v_cache: bf16 [num_pages, 16, H, D]
 *   (page id = physical 128-token block * 8 + page, as the table writes it);
 *   all three 16-byte aligned; D in {64, 128, 256}; 1 <= G <=
 *   BSA_MAX_ATTN_GROUP.  sparse_bt: int32 [T, H, K * 8]; sparse_ctx: int32
 *   [T, H]; out: fp32 [T, H, G, D].
 * Errors: BSA_ERR_NULL, BSA_ERR_SHAPE, BSA_ERR_TOPK (K < 1 or > BSA_MAX_TOPK),
 * BSA_ERR_ALIGN. */
int bsa_sparse_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                int64_t num_pages, const int32_t* sparse_bt,
                                const int32_t* sparse_ctx, int64_t T, int64_t H, int64_t G,
                                int64_t D, int32_t K, float scale, float* out, void* stream);

/* Size of the device scratch array behind bsa_topk_select_noalloc. */
#define BSA_NOALLOC_SCRATCH_BYTES (16u << 20)

/* bsa_topk_select for callers that cannot allocate device memory (no
 * counterpart on the pages: it exists for deployment, not for the method).
 * Same arguments, results and errors as bsa_topk_select, without the
 * workspace: when the launch policy needs one (few long rows), the library
 * uses a file-scope device array of BSA_NOALLOC_SCRATCH_BYTES (16 MiB) that
 * every GPU loading the library holds until the process exits.  Allocates
 * nothing.  Returns BSA_ERR_CAPACITY, before launching anything, when
 * bsa_topk_workspace_bytes(T, H, M, K, dtype) exceeds that size.  The first
 * call on a device, whether or not it needs scratch, looks the array's
 * address up (cudaGetSymbolAddress), so it should come before any stream
 * capture.  All calls on a device share the array: calls that overlap on the
 * GPU race.  out_idx is token-major int32[T, H, K]. */
int bsa_topk_select_noalloc(const void* scores, int32_t dtype, int64_t T, int64_t H, int64_t M,
                            int64_t token_stride, int64_t head_stride,
                            const int32_t* num_valid_pages, int32_t K, int32_t num_init,
                            int32_t num_local, int32_t* out_idx, void* stream);

/* The selector's launch policy ([55235] _decode_topk_launch_policy, redone
 * for sm_103a) for `rows` = T*H rows of capacity M on a GPU with `num_sms`
 * SMs.  Host-only, deterministic, launches nothing; exported so the 74 /
 * 128 / 129 and other capacity boundaries can be tested without a GPU.
 * Paths: BSA_PATH_PAIR when K <= 32 and a row holds at most 2 KB (M * element
 * size <= 2048), BSA_PATH_OCTET when 32 < K <= 64 and a row holds at most
 * 2 KB; BSA_PATH_SPLIT when a row needs more than one pass and the rows
 * alone cannot fill the GPU (at most num_sms * 16 rows); otherwise, for rows
 * of more than 2 KB (bf16 M > 1024, fp32 M > 512, up to the 8192-tile
 * capture-time capacity and beyond) with K <= 64, BSA_PATH_PAIR or BSA_PATH_OCTET with
 * long_rows = 1: those paths take every row whose non-forced range fits in
 * 2 KB and list the others, which a second launch on the same stream takes
 * with the wide path (one warp per row); BSA_PATH_ROW for the rest.  The
 * environment variable BSA_SELECT_PATH=row|group|pair|octet|wide, read once
 * per process, forces a path among those that can serve the call, for
 * testing (BSA_PATH_GROUP is reachable only that way; BSA_PATH_WIDE alone
 * takes every row with one warp).
 * Errors: BSA_ERR_NULL, BSA_ERR_SHAPE, BSA_ERR_TOPK, BSA_ERR_DTYPE. */
int bsa_select_policy(int64_t rows, int64_t M, int32_t K, int32_t dtype, int32_t num_sms,
                      bsa_launch_policy_t* policy);

/* ---- device status word ------------------------------------------------ */
/* A diagnostic aid of this library (the pages describe none; their kernels
 * mask the cases below, [47984] 实现拆解 item 3).  Instead of trapping, the
 * kernels set bits in a 32-bit device word that the caller registers when
 * they meet input that the calls above handle without a fault but that is
 * not valid:
 *   BSA_STATUS_BAD_BLOCK_ID  the sparse-table expansion (bsa_build_sparse_block_table
 *                            and the fused calls) met a block_table entry of a
 *                            kept block that is negative or above
 *                            BSA_MAX_PHYS_BLOCK (its page ids phys * 8 + p are
 *                            still written as computed); or the index scoring
 *                            met an entry of a causal block below max_blocks
 *                            outside [0, num_phys_blocks) (scored -inf).
 *   BSA_STATUS_BAD_PAGE      the sparse decode attention met a table entry of
 *                            a context token outside [0, num_pages) (the token
 *                            takes no part).
 *   BSA_STATUS_BAD_CONTEXT   the sparse decode attention met a sparse_ctx
 *                            entry below 0 or above K * 128 (clamped). */
#define BSA_STATUS_BAD_BLOCK_ID 0x1u
#define BSA_STATUS_BAD_PAGE 0x2u
#define BSA_STATUS_BAD_CONTEXT 0x4u
#define BSA_MAX_PHYS_BLOCK 0x0FFFFFFF  /* largest block id whose page ids fit int32 */

/* Registers `word`, a DEVICE pointer to one uint32 on the current device
 * (4-byte aligned, owned by the caller, zeroed by the caller), as that
 * device's status word; NULL unregisters it.  Calls made afterwards on the
 * device pass it to their kernels (a CUDA graph keeps the word registered
 * when it was captured); with none registered the kernels skip the checks.
 * Registration is not ordered against calls being made from other threads.
 * Errors: BSA_ERR_ALIGN; BSA_ERR_SHAPE for a device ordinal >= 64; a
 * positive cudaError_t when the current device cannot be read. */
int bsa_set_status_word(uint32_t* word);

/* Copies the current device's status word to *out (HOST) once the work
 * queued on `stream` so far is done, and clears the word when `clear` is
 * nonzero; synchronizes `stream`.  *out = 0 when no word is registered.
 * Errors: BSA_ERR_NULL (out); a positive cudaError_t from the copy. */
int bsa_read_status(uint32_t* out, int32_t clear, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BSA_TOPK_H_ */
