/*
 * bsa_oracle.c -- plain, slow, single-threaded CPU oracle for the block-sparse
 * attention top-k selection path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the CPU-baseline leg of the benchmark load this library.  The product path
 * (the CUDA library under block_sparse_attention_topk_gb300/) never links,
 * imports or calls it, and shares no code, header, table or helper with it.
 *
 * Everything here is the plain definition written out, in the order the
 * pages state it, with library sorts (qsort) as the only building block:
 *
 *  - causal page bound: "vLLM PR #47502 report" ([Minimax-M3] Using
 *    tok_sparse_select from MSA instead of triton kernels), section
 *    关键源码片段, indexer_msa.py: the metadata holds, per token row, the
 *    number of 128-token pages covering positions 0 .. pos, and the module
 *    docstring bounds each row by that count, always keeps the init and local
 *    blocks, and fills the unwritten tail with -inf.
 *  - total order incl. NaN, +-Inf, +-0 and ties: "vLLM PR #55235 report"
 *    ([ROCm][Perf] Tune MiniMax-M3 decode top-k for short contexts), sections
 *    执行摘要 and 评论区精华 (independent CPU total-order reference).  The
 *    order used is IEEE 754-2019 clause 5.10 totalOrder; ties between equal
 *    bit patterns go to the lower block id.
 *  - decode row mapping, padded rows and the hardened validity mask of the
 *    sparse block table: "vLLM PR #47984 report" ([ROCm][MiniMax-M3][Spec
 *    Decode] Support speculative decode with AITER sparse PA), sections
 *    实现拆解 items 1 and 3 and 关键源码片段 (the test loop and
 *    minimax_m3_build_sparse_block_table_decode).
 *
 * Readings taken where the pages are silent (each is listed with its reason
 * in the design notes): output slots hold the selected ids in ascending
 * block-id order followed by -1; "local" blocks are the last num_local causal
 * blocks [v-L, v); init blocks are [0, I); the sparse table lists the valid,
 * distinct selected blocks in ascending id order, 8 page-16 entries each,
 * with pages that start at or after the causal length left 0; ids that are
 * negative, >= the causal page count, or >= the block-table width are
 * ignored; a repeated id counts once.
 *
 * The floating-point inputs are only compared, never combined, so there is
 * no rounding anywhere in this file: bf16 and fp32 bit patterns are decoded
 * exactly into doubles (ldexp of an integer mantissa) for the numeric part
 * of totalOrder.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_PAGE_SIZE 128            /* tokens per sparse block / page    */
#define ORACLE_SUB_PAGE 16              /* tokens per page-16 table entry    */
#define ORACLE_PAGES_PER_BLOCK (ORACLE_PAGE_SIZE / ORACLE_SUB_PAGE)

enum { ORACLE_BF16 = 0, ORACLE_FP32 = 1 };

/* ------------------------------------------------------------------------ */
/* IEEE 754 decoding and totalOrder                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
    int is_nan;        /* exponent all ones, fraction non-zero            */
    int negative;      /* sign bit                                         */
    uint32_t payload;  /* fraction field of a NaN (quiet bit included)     */
    double value;      /* exact numeric value when not NaN (+-0 kept)      */
} decoded_t;

/* Decode a binary floating-point bit pattern with `ebits` exponent bits and
 * `fbits` fraction bits (bf16: 8/7, fp32: 8/23). */
static decoded_t decode_bits(uint32_t bits, int ebits, int fbits) {
    decoded_t d;
    const uint32_t fmask = (1u << fbits) - 1u;
    const uint32_t emask = (1u << ebits) - 1u;
    const int bias = (int)(emask >> 1);
    uint32_t frac = bits & fmask;
    uint32_t expo = (bits >> fbits) & emask;
    d.negative = (int)((bits >> (fbits + ebits)) & 1u);
    d.is_nan = (expo == emask) && (frac != 0);
    d.payload = d.is_nan ? frac : 0;
    if (expo == emask) {
        d.value = frac ? NAN : INFINITY;
    } else if (expo == 0) {
        /* zero or subnormal: frac * 2^(1 - bias - fbits) */
        d.value = ldexp((double)frac, 1 - bias - fbits);
    } else {
        d.value = ldexp((double)(frac | (1u << fbits)), (int)expo - bias - fbits);
    }
    if (d.negative && !d.is_nan) d.value = -d.value;
    return d;
}

static decoded_t decode_score(const void* base, int dtype, int64_t index) {
    if (dtype == ORACLE_BF16) {
        uint16_t b;
        memcpy(&b, (const char*)base + index * 2, 2);
        return decode_bits(b, 8, 7);
    }
    uint32_t b;
    memcpy(&b, (const char*)base + index * 4, 4);
    return decode_bits(b, 8, 23);
}

/* IEEE 754-2019 5.10 totalOrder, as a three-way comparison.
 *  - a NaN with the sign bit set is below every non-NaN, one without it above;
 *  - among NaNs of the same sign, signalling orders below quiet for positive
 *    NaNs and above for negative ones; the remaining payload order is
 *    implementation-defined, and here a larger fraction field lies further
 *    from zero (which also realises the signalling/quiet rule, because the
 *    quiet bit is the top fraction bit);
 *  - numbers compare by value, and -0 is below +0. */
static int total_order_cmp(decoded_t a, decoded_t b) {
    if (a.is_nan || b.is_nan) {
        if (a.is_nan && b.is_nan) {
            if (a.negative != b.negative) return a.negative ? -1 : 1;
            if (a.payload == b.payload) return 0;
            int a_smaller = a.payload < b.payload;
            if (a.negative) return a_smaller ? 1 : -1;
            return a_smaller ? -1 : 1;
        }
        if (a.is_nan) return a.negative ? -1 : 1;
        return b.negative ? 1 : -1;
    }
    if (a.value < b.value) return -1;
    if (a.value > b.value) return 1;
    if (a.value == 0.0 && a.negative != b.negative) return a.negative ? -1 : 1;
    return 0;
}

int oracle_total_order_cmp(uint32_t a_bits, uint32_t b_bits, int dtype) {
    if (dtype == ORACLE_BF16)
        return total_order_cmp(decode_bits(a_bits & 0xFFFFu, 8, 7),
                               decode_bits(b_bits & 0xFFFFu, 8, 7));
    return total_order_cmp(decode_bits(a_bits, 8, 23), decode_bits(b_bits, 8, 23));
}

/* ------------------------------------------------------------------------ */
/* Causal page bound                                                          */
/* ------------------------------------------------------------------------ */

/* Pages of 128 tokens needed to hold a causal prefix of `len` tokens. */
static int32_t pages_for_length(int64_t len) {
    if (len <= 0) return 0;
    return (int32_t)((len + ORACLE_PAGE_SIZE - 1) / ORACLE_PAGE_SIZE);
}

/* Decode rows: row = req*dql + local_q, query position
 * seq_len[req] - dql + local_q, causal length position + 1 (0 when the
 * position is negative, e.g. padded requests with seq_len 0). */
int oracle_num_valid_pages_decode(const int32_t* seq_lens, int64_t num_reqs,
                                  int32_t dql, int32_t* out) {
    if (dql < 1) return -1;
    for (int64_t req = 0; req < num_reqs; ++req) {
        for (int32_t q = 0; q < dql; ++q) {
            int64_t pos = (int64_t)seq_lens[req] - dql + q;
            int64_t causal_len = pos + 1 > 0 ? pos + 1 : 0;
            out[req * dql + q] = pages_for_length(causal_len);
        }
    }
    return 0;
}

/* Varlen rows: sequence i owns rows [cu[i], cu[i+1]); its j-th query token
 * sits at position prefix_lens[i] + j. */
int oracle_num_valid_pages_varlen(const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                                  int64_t num_seqs, int32_t* out) {
    for (int64_t i = 0; i < num_seqs; ++i) {
        for (int64_t row = cu_seqlens_q[i]; row < cu_seqlens_q[i + 1]; ++row) {
            int64_t pos = (int64_t)prefix_lens[i] + (row - cu_seqlens_q[i]);
            out[row] = pages_for_length(pos + 1);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Top-k selection                                                            */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t id;
    int forced;
    decoded_t score;
} entry_t;

/* "Better first": forced blocks, then higher totalOrder, then lower id. */
static int entry_better_first(const void* pa, const void* pb) {
    const entry_t* a = (const entry_t*)pa;
    const entry_t* b = (const entry_t*)pb;
    if (a->forced != b->forced) return a->forced ? -1 : 1;
    int c = total_order_cmp(a->score, b->score);
    if (c != 0) return -c;
    return (a->id > b->id) - (a->id < b->id);
}

static int int32_ascending(const void* pa, const void* pb) {
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a > b) - (a < b);
}

/* scores: element (t, h, b) at scores[t*token_stride + h*head_stride + b]
 * nvp:    int32[T] causal page counts
 * out:    int32[T, H, K] token-major; ascending selected ids, then -1. */
int oracle_topk_select(const void* scores, int dtype, int64_t T, int64_t H, int64_t M,
                       int64_t token_stride, int64_t head_stride, const int32_t* nvp,
                       int32_t K, int32_t num_init, int32_t num_local, int32_t* out) {
    if (K < 1 || num_init < 0 || num_local < 0) return -1;
    entry_t* entries = (entry_t*)malloc(sizeof(entry_t) * (size_t)(M > 0 ? M : 1));
    int32_t* chosen = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
    if (!entries || !chosen) { free(entries); free(chosen); return -2; }
    for (int64_t t = 0; t < T; ++t) {
        int64_t v = nvp[t] < M ? nvp[t] : M;
        if (v < 0) v = 0;
        for (int64_t h = 0; h < H; ++h) {
            int32_t* dst = out + (t * H + h) * K;
            int64_t row = t * token_stride + h * head_stride;
            for (int64_t b = 0; b < v; ++b) {
                entries[b].id = (int32_t)b;
                entries[b].forced = (b < num_init) || (b >= v - num_local);
                entries[b].score = decode_score(scores, dtype, row + b);
            }
            qsort(entries, (size_t)v, sizeof(entry_t), entry_better_first);
            int64_t n = v < K ? v : K;
            for (int64_t i = 0; i < n; ++i) chosen[i] = entries[i].id;
            qsort(chosen, (size_t)n, sizeof(int32_t), int32_ascending);
            for (int64_t i = 0; i < K; ++i) dst[i] = i < n ? chosen[i] : -1;
        }
    }
    free(entries);
    free(chosen);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Sparse block table (page-16 rows)                                          */
/* ------------------------------------------------------------------------ */

/* topk_idx:    int32[T, H, K] (any ids; -1 and out-of-range ids ignored)
 * block_table: int32[B, MB] physical 128-token block ids per request
 * seq_lens:    int32[B]; T = B * dql
 * sparse_bt:   int32[T, H, K*8]; sparse_ctx: int32[T, H] */
int oracle_build_sparse_block_table(const int32_t* topk_idx, int64_t T, int64_t H, int32_t K,
                                    const int32_t* block_table, int64_t B, int64_t MB,
                                    const int32_t* seq_lens, int32_t dql,
                                    int32_t* sparse_bt, int32_t* sparse_ctx) {
    if (dql < 1 || T != B * dql || K < 1) return -1;
    int32_t* blocks = (int32_t*)malloc(sizeof(int32_t) * (size_t)K);
    if (!blocks) return -2;
    const int64_t width = (int64_t)K * ORACLE_PAGES_PER_BLOCK;
    for (int64_t r = 0; r < T; ++r) {
        int64_t req = r / dql;
        int64_t local_q = r % dql;
        int64_t pos = (int64_t)seq_lens[req] - dql + local_q;
        int64_t causal_len = pos + 1 > 0 ? pos + 1 : 0;
        int64_t num_blocks = pages_for_length(causal_len);
        for (int64_t h = 0; h < H; ++h) {
            const int32_t* ids = topk_idx + (r * H + h) * K;
            int32_t* bt = sparse_bt + (r * H + h) * width;
            int64_t n = 0;
            for (int32_t i = 0; i < K; ++i) {
                int32_t b = ids[i];
                if (b < 0 || b >= num_blocks || b >= MB) continue;
                int dup = 0;
                for (int64_t j = 0; j < n; ++j) dup |= blocks[j] == b;
                if (!dup) blocks[n++] = b;
            }
            qsort(blocks, (size_t)n, sizeof(int32_t), int32_ascending);
            for (int64_t e = 0; e < width; ++e) bt[e] = 0;
            int64_t ctx = 0;
            for (int64_t j = 0; j < n; ++j) {
                int64_t b = blocks[j];
                int32_t phys = block_table[req * MB + b];
                for (int p = 0; p < ORACLE_PAGES_PER_BLOCK; ++p) {
                    if (b * ORACLE_PAGE_SIZE + (int64_t)p * ORACLE_SUB_PAGE < causal_len)
                        bt[j * ORACLE_PAGES_PER_BLOCK + p] = phys * ORACLE_PAGES_PER_BLOCK + p;
                }
                int64_t tokens = causal_len - b * ORACLE_PAGE_SIZE;
                ctx += tokens < ORACLE_PAGE_SIZE ? tokens : ORACLE_PAGE_SIZE;
            }
            sparse_ctx[r * H + h] = (int32_t)ctx;
        }
    }
    free(blocks);
    return 0;
}

/* Select-then-expand for decode rows, as one call: the definition of the
 * fused selector with the sparse-table epilogue is exactly the composition
 * of the two steps above (the fused kernel only avoids the round trip). */
int oracle_topk_select_sparse_table(const void* scores, int dtype, int64_t B, int32_t dql,
                                    int64_t H, int64_t M, int64_t token_stride,
                                    int64_t head_stride, const int32_t* seq_lens, int32_t K,
                                    int32_t num_init, int32_t num_local,
                                    const int32_t* block_table, int64_t MB, int32_t* out_idx,
                                    int32_t* sparse_bt, int32_t* sparse_ctx) {
    int64_t T = B * dql;
    int32_t* nvp = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    if (!nvp) return -2;
    int rc = oracle_num_valid_pages_decode(seq_lens, B, dql, nvp);
    if (rc == 0)
        rc = oracle_topk_select(scores, dtype, T, H, M, token_stride, head_stride, nvp, K,
                                num_init, num_local, out_idx);
    if (rc == 0)
        rc = oracle_build_sparse_block_table(out_idx, T, H, K, block_table, B, MB, seq_lens,
                                             dql, sparse_bt, sparse_ctx);
    free(nvp);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Index scores of decode rows                                                */
/* ------------------------------------------------------------------------ */

/* The pages name the decode score kernel (minimax_m3_index_decode_score,
 * writing score_out = unified_scores[:nd]: "vLLM PR #47502 report", section
 * 实现拆解 item 1) and say that a page, a sparse block and an index-K block
 * are the same 128 tokens (section 关键源码片段, indexer_msa.py), but they do
 * not print the score formula.  Reading taken: one pooled index key per
 * physical 128-token block, shared by the index heads, and
 *     score[t, h, b] = sum over d of q[t, h, d] * k[block_table[req, b], d]
 * with req = t / dql (the decode row mapping of PR #47984), no scale factor
 * (PR #47502 removed sm_scale from the top-k call: section 实现拆解 item 6),
 * computed here exactly (bf16 products are exact in double, and the sum of
 * D of them is rounded once per addition in double).  Only the causal blocks
 * b < v = min(M, cdiv(pos + 1, 128)) have a score; a causal block without a
 * usable key (b >= MB, or a physical id outside [0, NB)) scores -inf, like
 * an unwritten tile.  Entries b >= v are set to NaN here: no score kernel
 * writes them.
 *
 * q: bf16 bits [T, H, D]; k: bf16 bits [NB, D]; block_table: int32 [B, MB];
 * seq_lens: int32 [B]; T = B * dql; out: double [T, H, M]. */
int oracle_index_scores(const uint16_t* q, const uint16_t* k, int64_t NB,
                        const int32_t* block_table, int64_t MB, const int32_t* seq_lens,
                        int64_t B, int32_t dql, int64_t H, int64_t D, int64_t M, double* out) {
    if (dql < 1 || H < 1 || D < 1 || M < 1) return -1;
    for (int64_t req = 0; req < B; ++req) {
        for (int32_t lq = 0; lq < dql; ++lq) {
            const int64_t t = req * dql + lq;
            const int64_t pos = (int64_t)seq_lens[req] - dql + lq;
            int64_t v = pages_for_length(pos + 1 > 0 ? pos + 1 : 0);
            if (v > M) v = M;
            for (int64_t h = 0; h < H; ++h) {
                double* row = out + (t * H + h) * M;
                const uint16_t* qv = q + (t * H + h) * D;
                for (int64_t b = 0; b < M; ++b) {
                    if (b >= v) {
                        row[b] = NAN;
                        continue;
                    }
                    const int64_t phys = b < MB ? block_table[req * MB + b] : -1;
                    if (phys < 0 || phys >= NB) {
                        row[b] = -INFINITY;
                        continue;
                    }
                    double s = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        s += decode_bits(qv[d], 8, 7).value * decode_bits(k[phys * D + d], 8, 7).value;
                    row[b] = s;
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Sparse decode attention over the page-16 table                            */
/* ------------------------------------------------------------------------ */

/* The consumer of the sparse table: "vLLM PR #47984 report", 实现拆解 items
 * 1-2 (the ROCm sparse paged-attention decode reads the page-16 table and
 * its sparse_ctx) and "vLLM PR #47502 report", 实现拆解 item 5 (the sparse
 * decode kernels count their valid blocks from the sequence position).  The
 * pages show the interface only.  Readings taken: index head h selects for
 * KV head h, which G query heads share; the KV cache is paged in 16-token
 * pages (bf16 [num_pages, 16, H, D], page id = physical 128-token block * 8
 * + page, as the table writes it); row (t, h) attends to its first
 * ctx = sparse_ctx[t, h] table tokens, token j sitting in page
 * sparse_bt[t, h, j / 16] at slot j % 16; and each query head g takes
 *     out[t, h, g] = sum_j softmax_j(scale * q[t, h, g] . k_j) v_j
 * in exact arithmetic (here double).  A row with an empty context yields
 * zeros; a token whose page id lies outside [0, num_pages) takes no part.
 *
 * q: bf16 [T, H, G, D]; k_cache, v_cache: bf16 [num_pages, 16, H, D];
 * sparse_bt: int32 [T, H, K * 8]; sparse_ctx: int32 [T, H];
 * out: double [T, H, G, D]. */
int oracle_sparse_decode_attention(const uint16_t* q, const uint16_t* k_cache,
                                   const uint16_t* v_cache, int64_t num_pages,
                                   const int32_t* sparse_bt, const int32_t* sparse_ctx,
                                   int64_t T, int64_t H, int64_t G, int64_t D, int32_t K,
                                   double scale, double* out) {
    if (T < 0 || H < 1 || G < 1 || D < 1 || K < 1) return -1;
    const int64_t width = (int64_t)K * ORACLE_PAGES_PER_BLOCK;
    double* s = (double*)malloc(sizeof(double) * (size_t)(width * ORACLE_SUB_PAGE));
    if (!s) return -2;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            const int32_t* bt = sparse_bt + (t * H + h) * width;
            int64_t ctx = sparse_ctx[t * H + h];
            if (ctx > width * ORACLE_SUB_PAGE) ctx = width * ORACLE_SUB_PAGE;
            for (int64_t g = 0; g < G; ++g) {
                const uint16_t* qv = q + ((t * H + h) * G + g) * D;
                double* o = out + ((t * H + h) * G + g) * D;
                for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
                double mx = -INFINITY;
                for (int64_t j = 0; j < ctx; ++j) {
                    const int64_t page = bt[j / ORACLE_SUB_PAGE];
                    s[j] = -INFINITY;
                    if (page < 0 || page >= num_pages) continue;
                    const uint16_t* kv = k_cache + ((page * ORACLE_SUB_PAGE + j % ORACLE_SUB_PAGE) * H + h) * D;
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        dot += decode_bits(qv[d], 8, 7).value * decode_bits(kv[d], 8, 7).value;
                    s[j] = scale * dot;
                    if (s[j] > mx) mx = s[j];
                }
                if (mx == -INFINITY) continue;   /* empty context: zeros */
                double sum = 0.0;
                for (int64_t j = 0; j < ctx; ++j) {
                    if (s[j] == -INFINITY) continue;
                    const double p = exp(s[j] - mx);
                    const int64_t page = bt[j / ORACLE_SUB_PAGE];
                    const uint16_t* vv = v_cache + ((page * ORACLE_SUB_PAGE + j % ORACLE_SUB_PAGE) * H + h) * D;
                    for (int64_t d = 0; d < D; ++d) o[d] += p * decode_bits(vv[d], 8, 7).value;
                    sum += p;
                }
                for (int64_t d = 0; d < D; ++d) o[d] /= sum;
            }
        }
    }
    free(s);
    return 0;
}
