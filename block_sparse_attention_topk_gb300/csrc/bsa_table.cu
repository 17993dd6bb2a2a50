// bsa_table.cu -- causal page counts and the page-16 sparse block table.
//
// Causal page count: vLLM PR #47502 report ("[Minimax-M3] Using
// tok_sparse_select from MSA instead of triton kernels"), section 关键源码片段,
// indexer_msa.py metadata: each token row gets the number of 128-token pages
// that cover its positions 0 .. pos, i.e. ceil((pos + 1) / 128); varlen rows
// take their positions from the batch-wide topk_cu_seqlens_q and
// topk_prefix_lens.
// Decode row mapping and the sparse table: vLLM PR #47984 report ("Support
// speculative decode with AITER sparse PA"), sections 实现拆解 items 1-3 and
// 关键源码片段: row = req*dql + local_q, query position
// seq_len[req] - dql + local_q, causal_len = max(pos + 1, 0); each kept
// 128-token block becomes 8 page-16 entries through the request's block
// table; ids outside [0, cdiv(causal_len, 128)) and -1 are ignored; padded
// rows give an empty context.
//
// Both kernels are tiny integer passes bound by memory latency.  For topk up
// to 32 the table builder gives each (token, head) row a segment of 16 or 32
// lanes, one id per lane: the block-table gather is issued as soon as the id
// is known, and overlaps a segmented bitonic sort of (id, lane) that brings
// duplicates together; kept ids are compacted through shared memory and each
// lane writes one 32-byte slot of the row.  For topk up to 64 a warp takes one
// row with two ids per lane and sorts them the same way.  Larger topk gives
// one warp to a row and deduplicates and sorts the ids in shared memory by
// counting ranks (K <= 1024 ids).
#include <cuda_runtime.h>
#include <stdint.h>

#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__global__ void nvp_decode_kernel(const int32_t* __restrict__ seq_lens, int64_t num_reqs,
                                  int32_t dql, int32_t* __restrict__ out) {
    const int64_t total = num_reqs * dql;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < total;
         r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t req = r / dql;
        const int64_t pos = (int64_t)__ldg(seq_lens + req) - dql + (r - req * dql);
        out[r] = pos >= 0 ? (int32_t)((pos + kPageSize) >> kLogPageSize) : 0;
    }
}

__global__ void nvp_varlen_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ prefix,
                                  int64_t num_seqs, int64_t total_q, int32_t* __restrict__ out) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < total_q;
         r += (int64_t)gridDim.x * blockDim.x) {
        int32_t pages = 0;
        if (num_seqs > 0 && r >= __ldg(cu) && r < __ldg(cu + num_seqs)) {
            // largest i with cu[i] <= r
            int64_t lo = 0, hi = num_seqs;  // cu[lo] <= r < cu[hi]
            while (hi - lo > 1) {
                const int64_t mid = (lo + hi) >> 1;
                if (__ldg(cu + mid) <= r) lo = mid;
                else hi = mid;
            }
            const int64_t pos = (int64_t)__ldg(prefix + lo) + (r - __ldg(cu + lo));
            pages = pos >= 0 ? (int32_t)((pos + kPageSize) >> kLogPageSize) : 0;
        }
        out[r] = pages;
    }
}

constexpr int kTableWarps = 4;

// Shared memory per warp: ids[K], first-occurrence flags[K], sorted[K].
__global__ void __launch_bounds__(kTableWarps * 32)
sparse_table_kernel(const int32_t* __restrict__ topk_idx, int64_t rows, int64_t H, int32_t K,
                    const int32_t* __restrict__ block_table, int64_t max_blocks,
                    const int32_t* __restrict__ seq_lens, int32_t dql,
                    int32_t* __restrict__ sparse_bt, int32_t* __restrict__ sparse_ctx,
                    uint32_t* status) {
    extern __shared__ int32_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int32_t* s_ids = smem + (size_t)warp * 3 * K;
    int32_t* s_first = s_ids + K;
    int32_t* s_sorted = s_first + K;
    const int width = K * kPagesPerBlock;
    for (int64_t row = (int64_t)blockIdx.x * kTableWarps + warp; row < rows;
         row += (int64_t)gridDim.x * kTableWarps) {
        const int64_t t = row / H;
        const int64_t req = t / dql;
        const int64_t pos = (int64_t)__ldg(seq_lens + req) - dql + (t - req * dql);
        const int64_t causal_len = pos + 1 > 0 ? pos + 1 : 0;
        const int64_t nblk = (causal_len + kPageSize - 1) >> kLogPageSize;
        const int64_t limit = nblk < max_blocks ? nblk : max_blocks;
        const int32_t* ids = topk_idx + row * K;
        for (int i = lane; i < K; i += 32) {
            const int32_t x = __ldg(ids + i);
            s_ids[i] = (x >= 0 && x < limit) ? x : -1;
        }
        __syncwarp();
        // first occurrence of each valid id
        for (int i = lane; i < K; i += 32) {
            const int32_t x = s_ids[i];
            bool first = x >= 0;
            for (int j = 0; j < i && first; ++j) first = s_ids[j] != x;
            s_first[i] = first ? 1 : 0;
        }
        __syncwarp();
        // rank = number of distinct valid ids below x; scatter to sorted order
        int count = 0;
        for (int i = lane; i < K; i += 32) {
            if (!s_first[i]) continue;
            const int32_t x = s_ids[i];
            int rank = 0;
            for (int j = 0; j < K; ++j) rank += (s_first[j] && s_ids[j] < x) ? 1 : 0;
            s_sorted[rank] = x;
            ++count;
        }
        const int n = __reduce_add_sync(kFull, count);
        __syncwarp();
        const int32_t* table = block_table + req * max_blocks;
        int32_t* bt = sparse_bt + row * (int64_t)width;
        for (int e = lane; e < width; e += 32) {
            const int j = e >> 3;
            const int pg = e & 7;
            int32_t val = 0;
            if (j < n) {
                const int32_t b = s_sorted[j];
                if ((int64_t)b * kPageSize + (int64_t)pg * kSubPage < causal_len) {
                    const int32_t phys = __ldg(table + b);
                    report_status(status, pg == 0 && bad_phys_block(phys), BSA_STATUS_BAD_BLOCK_ID);
                    val = phys * kPagesPerBlock + pg;
                }
            }
            bt[e] = val;
        }
        int ctx = 0;
        for (int j = lane; j < n; j += 32) {
            const int64_t rem = causal_len - (int64_t)s_sorted[j] * kPageSize;
            ctx += (int)(rem < kPageSize ? rem : kPageSize);
        }
        ctx = __reduce_add_sync(kFull, ctx);
        if (lane == 0) sparse_ctx[row] = ctx;
        __syncwarp();
    }
}

// topk <= 32: G lanes per row (G = 16 for K <= 16, else 32), 32 / G rows per
// warp.  VEC: the output table is 32-byte aligned, so each slot is written
// with one 256-bit store.
constexpr int kSegWarps = 8;

template <int G, bool VEC>
__global__ void __launch_bounds__(kSegWarps * 32)
sparse_table_seg_kernel(const int32_t* __restrict__ topk_idx, int64_t rows, int64_t H, int32_t K,
                        const int32_t* __restrict__ block_table, int64_t max_blocks,
                        const int32_t* __restrict__ seq_lens, int32_t dql,
                        int32_t* __restrict__ sparse_bt, int32_t* __restrict__ sparse_ctx,
                        uint32_t* status) {
    constexpr int R = 32 / G;                  // rows per warp
    constexpr int32_t kNone = 0x7FFFFFFF;      // sorts after every (id << 5 | lane)
    __shared__ int32_t s_blk[kSegWarps][32];
    __shared__ int32_t s_phys[kSegWarps][32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane & (G - 1);              // lane within the row's segment
    const int seg = lane - g;                  // first lane of the segment
    const int width = K * kPagesPerBlock;
    for (int64_t base = ((int64_t)blockIdx.x * kSegWarps + warp) * R; base < rows;
         base += (int64_t)gridDim.x * kSegWarps * R) {
        const int64_t row = base + lane / G;
        const bool active = row < rows;
        int64_t causal_len = 0;
        int32_t key = kNone;
        int32_t phys = 0;
        if (active) {
            const int64_t t = row / H;
            const int64_t req = t / dql;
            const int64_t pos = (int64_t)__ldg(seq_lens + req) - dql + (t - req * dql);
            causal_len = pos + 1 > 0 ? pos + 1 : 0;
            const int64_t nblk = (causal_len + kPageSize - 1) >> kLogPageSize;
            const int64_t limit = nblk < max_blocks ? nblk : max_blocks;
            if (g < K) {
                const int32_t x = __ldg(topk_idx + row * K + g);
                if (x >= 0 && x < limit) {
                    key = (x << 5) | lane;
                    phys = __ldg(block_table + req * max_blocks + x);
                }
            }
        }
        // ascending bitonic sort of the segment's keys; equal ids end up
        // adjacent, ordered by lane
#pragma unroll
        for (int k = 2; k <= G; k <<= 1) {
#pragma unroll
            for (int j = k >> 1; j > 0; j >>= 1) {
                const int32_t other = __shfl_xor_sync(kFull, key, j);
                const bool take_min = ((g & j) == 0) == ((g & k) == 0 || k == G);
                key = take_min ? min(key, other) : max(key, other);
            }
        }
        const int32_t prev = __shfl_up_sync(kFull, key, 1);
        const bool keep = key != kNone && (g == 0 || (prev >> 5) != (key >> 5));
        // the gathered entry travels from the lane that loaded it
        const int32_t got = __shfl_sync(kFull, phys, key & 31);
        const unsigned segmask = G == 32 ? kFull : (0xFFFFu << seg);
        const unsigned kept = __ballot_sync(kFull, keep) & segmask;
        const int n = __popc(kept);
        if (keep) {
            const int rank = __popc(kept & ((1u << lane) - 1u));
            s_blk[warp][seg + rank] = key >> 5;
            s_phys[warp][seg + rank] = got;
        }
        __syncwarp();
        int32_t contrib = 0;
        if (active && g < K) {
            int32_t v[8];
            if (g < n) {
                const int32_t b = s_blk[warp][lane];
                const int32_t ph = s_phys[warp][lane];
                report_status(status, bad_phys_block(ph), BSA_STATUS_BAD_BLOCK_ID);
                const int64_t first = (int64_t)b * kPageSize;
#pragma unroll
                for (int pg = 0; pg < 8; ++pg)
                    v[pg] = first + pg * kSubPage < causal_len ? ph * kPagesPerBlock + pg : 0;
                const int64_t rem = causal_len - first;
                contrib = (int32_t)(rem < kPageSize ? rem : kPageSize);
            } else {
#pragma unroll
                for (int pg = 0; pg < 8; ++pg) v[pg] = 0;
            }
            int32_t* dst = sparse_bt + row * (int64_t)width + g * kPagesPerBlock;
            if constexpr (VEC) {
                st_v8(dst, v);
            } else {
#pragma unroll
                for (int pg = 0; pg < 8; ++pg) dst[pg] = v[pg];
            }
        }
#pragma unroll
        for (int off = G >> 1; off > 0; off >>= 1) contrib += __shfl_xor_sync(kFull, contrib, off);
        if (active && g == 0) sparse_ctx[row] = contrib;
        __syncwarp();
    }
}

// 32 < topk <= 64: one warp per row, two ids per lane.  Element e = 2 * lane
// + h (h = 0, 1) holds id e of the row; the 64 keys (id << 6 | e) are sorted
// across the warp with a bitonic network whose last stage compares a lane's
// own two registers.  Ids are below cdiv(seq_len, 128) <= 2^24, so the key
// does not overflow.
template <bool VEC>
__global__ void __launch_bounds__(kSegWarps * 32)
sparse_table_seg64_kernel(const int32_t* __restrict__ topk_idx, int64_t rows, int64_t H,
                          int32_t K, const int32_t* __restrict__ block_table,
                          int64_t max_blocks, const int32_t* __restrict__ seq_lens, int32_t dql,
                          int32_t* __restrict__ sparse_bt, int32_t* __restrict__ sparse_ctx,
                        uint32_t* status) {
    constexpr int32_t kNone = 0x7FFFFFFF;      // sorts after every (id << 6 | e)
    __shared__ int32_t s_in[kSegWarps][64];    // gathered entry by element
    __shared__ int32_t s_blk[kSegWarps][64];   // kept ids, ascending
    __shared__ int32_t s_phys[kSegWarps][64];  // their gathered entries
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int width = K * kPagesPerBlock;
    for (int64_t row = (int64_t)blockIdx.x * kSegWarps + warp; row < rows;
         row += (int64_t)gridDim.x * kSegWarps) {
        const int64_t t = row / H;
        const int64_t req = t / dql;
        const int64_t pos = (int64_t)__ldg(seq_lens + req) - dql + (t - req * dql);
        const int64_t causal_len = pos + 1 > 0 ? pos + 1 : 0;
        const int64_t nblk = (causal_len + kPageSize - 1) >> kLogPageSize;
        const int64_t limit = nblk < max_blocks ? nblk : max_blocks;
        const int32_t* table = block_table + req * max_blocks;
        int32_t key[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = 2 * lane + h;
            key[h] = kNone;
            int32_t phys = 0;
            if (e < K) {
                const int32_t x = __ldg(topk_idx + row * K + e);
                if (x >= 0 && x < limit) {
                    key[h] = (x << 6) | e;
                    phys = __ldg(table + x);
                }
            }
            s_in[warp][e] = phys;
        }
        // ascending bitonic sort of the 64 keys; equal ids end up adjacent,
        // ordered by element
#pragma unroll
        for (int k = 2; k <= 64; k <<= 1) {
            const bool asc = k == 64 || (lane & (k >> 1)) == 0;
#pragma unroll
            for (int j = k >> 1; j > 1; j >>= 1) {
                const bool take_min = ((lane & (j >> 1)) == 0) == asc;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int32_t other = __shfl_xor_sync(kFull, key[h], j >> 1);
                    key[h] = take_min ? min(key[h], other) : max(key[h], other);
                }
            }
            const int32_t lo = min(key[0], key[1]);
            const int32_t hi = max(key[0], key[1]);
            key[0] = asc ? lo : hi;
            key[1] = asc ? hi : lo;
        }
        const int32_t prev1 = __shfl_up_sync(kFull, key[1], 1);
        const bool keep0 = key[0] != kNone && (lane == 0 || (prev1 >> 6) != (key[0] >> 6));
        const bool keep1 = key[1] != kNone && (key[0] >> 6) != (key[1] >> 6);
        const unsigned b0 = __ballot_sync(kFull, keep0);
        const unsigned b1 = __ballot_sync(kFull, keep1);
        const int n = __popc(b0) + __popc(b1);
        __syncwarp();
        const unsigned below = (1u << lane) - 1u;
        const int rank0 = __popc(b0 & below) + __popc(b1 & below);
        if (keep0) {
            s_blk[warp][rank0] = key[0] >> 6;
            s_phys[warp][rank0] = s_in[warp][key[0] & 63];
        }
        if (keep1) {
            const int rank1 = rank0 + (keep0 ? 1 : 0);
            s_blk[warp][rank1] = key[1] >> 6;
            s_phys[warp][rank1] = s_in[warp][key[1] & 63];
        }
        __syncwarp();
        int32_t contrib = 0;
        int32_t* out = sparse_bt + row * (int64_t)width;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int j = lane + 32 * u;
            if (j >= K) continue;
            int32_t v[8];
            if (j < n) {
                const int32_t b = s_blk[warp][j];
                const int32_t ph = s_phys[warp][j];
                report_status(status, bad_phys_block(ph), BSA_STATUS_BAD_BLOCK_ID);
                const int64_t first = (int64_t)b * kPageSize;
#pragma unroll
                for (int pg = 0; pg < 8; ++pg)
                    v[pg] = first + pg * kSubPage < causal_len ? ph * kPagesPerBlock + pg : 0;
                const int64_t rem = causal_len - first;
                contrib += (int32_t)(rem < kPageSize ? rem : kPageSize);
            } else {
#pragma unroll
                for (int pg = 0; pg < 8; ++pg) v[pg] = 0;
            }
            int32_t* dst = out + j * kPagesPerBlock;
            if constexpr (VEC) {
                st_v8(dst, v);
            } else {
#pragma unroll
                for (int pg = 0; pg < 8; ++pg) dst[pg] = v[pg];
            }
        }
        contrib = __reduce_add_sync(kFull, contrib);
        if (lane == 0) sparse_ctx[row] = contrib;
        __syncwarp();
    }
}

int grid_for(int64_t work, int per_block, int max_blocks_per_sm) {
    int64_t g = (work + per_block - 1) / per_block;
    const int64_t cap = (int64_t)device_sm_count() * max_blocks_per_sm;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_num_valid_pages_decode(const int32_t* seq_lens, int64_t num_reqs, int32_t dql,
                                          int32_t* out, cudaStream_t stream) {
    const int64_t total = num_reqs * dql;
    if (total == 0) return cudaSuccess;
    nvp_decode_kernel<<<grid_for(total, 256, 8), 256, 0, stream>>>(seq_lens, num_reqs, dql, out);
    return cudaGetLastError();
}

cudaError_t launch_num_valid_pages_varlen(const int32_t* cu, const int32_t* prefix,
                                          int64_t num_seqs, int64_t total_q, int32_t* out,
                                          cudaStream_t stream) {
    if (total_q == 0) return cudaSuccess;
    nvp_varlen_kernel<<<grid_for(total_q, 256, 8), 256, 0, stream>>>(cu, prefix, num_seqs,
                                                                     total_q, out);
    return cudaGetLastError();
}

cudaError_t launch_build_sparse_block_table(const int32_t* topk_idx, int64_t T, int64_t H,
                                            int32_t K, const int32_t* block_table,
                                            int64_t max_blocks, const int32_t* seq_lens,
                                            int32_t dql, int32_t* sparse_bt,
                                            int32_t* sparse_ctx, cudaStream_t stream) {
    const int64_t rows = T * H;
    if (rows == 0) return cudaSuccess;
    uint32_t* status = current_status_word();
    if (K <= 32) {
        const bool vec = (reinterpret_cast<uintptr_t>(sparse_bt) & 31) == 0;
        const int per_block = kSegWarps * (K <= 16 ? 2 : 1);
        // one row group per warp, grid not capped at the resident CTAs
        const int grid = grid_for(rows, per_block, 1 << 20);
        auto kern = K <= 16 ? (vec ? sparse_table_seg_kernel<16, true>
                                   : sparse_table_seg_kernel<16, false>)
                            : (vec ? sparse_table_seg_kernel<32, true>
                                   : sparse_table_seg_kernel<32, false>);
        kern<<<grid, kSegWarps * 32, 0, stream>>>(topk_idx, rows, H, K, block_table, max_blocks,
                                                  seq_lens, dql, sparse_bt, sparse_ctx, status);
        return cudaGetLastError();
    }
    if (K <= 64) {
        const bool vec = (reinterpret_cast<uintptr_t>(sparse_bt) & 31) == 0;
        // one row per warp, grid not capped at the resident CTAs
        const int grid = grid_for(rows, kSegWarps, 1 << 20);
        auto kern = vec ? sparse_table_seg64_kernel<true> : sparse_table_seg64_kernel<false>;
        kern<<<grid, kSegWarps * 32, 0, stream>>>(topk_idx, rows, H, K, block_table, max_blocks,
                                                  seq_lens, dql, sparse_bt, sparse_ctx, status);
        return cudaGetLastError();
    }
    const size_t smem = (size_t)kTableWarps * 3 * K * sizeof(int32_t);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(sparse_table_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    sparse_table_kernel<<<grid_for(rows, kTableWarps, 16), kTableWarps * 32, smem, stream>>>(
        topk_idx, rows, H, K, block_table, max_blocks, seq_lens, dql, sparse_bt, sparse_ctx, status);
    return cudaGetLastError();
}

}  // namespace bsa
