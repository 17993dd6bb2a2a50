// bsa_capi.cu -- the extern "C" entry points declared in include/bsa_topk.h:
// host-side argument checks, the launch policy and the workspace carve-up.
// Every compute step runs in the kernels of bsa_select.cu and bsa_table.cu.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <climits>
#include <mutex>

#include "bsa_internal.h"

namespace bsa {

namespace {
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];
std::once_flag g_sm_once[kMaxDevices];
std::atomic<uint32_t*> g_status_word[kMaxDevices];

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int elem_bytes(int32_t dtype) { return dtype == BSA_DTYPE_BF16 ? 2 : 4; }
}  // namespace

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 152;
    std::call_once(g_sm_once[dev], [dev] {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        g_sm_count[dev] = n;
    });
    return g_sm_count[dev];
}

uint32_t* current_status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    return g_status_word[dev].load(std::memory_order_acquire);
}

size_t split_workspace_bytes(int64_t rows, int32_t chunks, int32_t K) {
    if (chunks <= 1 || rows <= 0) return 0;
    const size_t entries = (size_t)rows * chunks * K;
    return align_up(entries * 4) + align_up(entries * 4) + align_up((size_t)rows * chunks * 4) +
           align_up((size_t)rows * 4);
}

// The list of rows left to the wide path and its counter.
size_t long_workspace_bytes(int64_t rows) { return align_up((size_t)rows * 4) + kAlign; }

size_t select_workspace_bytes(int64_t rows, const bsa_launch_policy_t& pol, int32_t K) {
    return pol.long_rows ? long_workspace_bytes(rows)
                         : split_workspace_bytes(rows, pol.chunks_per_row, K);
}

SplitWorkspace carve_split_workspace(void* base, int64_t rows, int32_t chunks, int32_t K) {
    SplitWorkspace ws{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    if (chunks <= 1 || base == nullptr) return ws;
    const size_t entries = (size_t)rows * chunks * K;
    char* p = static_cast<char*>(base);
    ws.keys = reinterpret_cast<uint32_t*>(p);
    p += align_up(entries * 4);
    ws.ids = reinterpret_cast<int32_t*>(p);
    p += align_up(entries * 4);
    ws.counts = reinterpret_cast<int32_t*>(p);
    p += align_up((size_t)rows * chunks * 4);
    ws.tickets = reinterpret_cast<int32_t*>(p);
    return ws;
}

}  // namespace bsa

using namespace bsa;

namespace {

int check_topk_args(int64_t M, int32_t K, int32_t num_init, int32_t num_local) {
    if (K < 1 || K > BSA_MAX_TOPK || K > M || num_init < 0 || num_local < 0 ||
        (int64_t)num_init + num_local > K)
        return BSA_ERR_TOPK;
    return BSA_OK;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? BSA_OK : (int)e; }

// Rows (t, h) of out_idx start at t * ots + h * ohs and hold K contiguous
// slots.  Accepted when no two rows can overlap: with the dimensions of more
// than one entry ordered by stride, the inner stride is at least K and the
// outer one clears the last inner row.
int check_out_layout(int64_t T, int64_t H, int32_t K, int64_t ots, int64_t ohs) {
    if (ots < 0 || ohs < 0) return BSA_ERR_SHAPE;
    int64_t n[2], st[2];
    int d = 0;
    if (T > 1) { n[d] = T; st[d] = ots; ++d; }
    if (H > 1) { n[d] = H; st[d] = ohs; ++d; }
    if (d == 1 && st[0] < K) return BSA_ERR_SHAPE;
    if (d == 2) {
        const int in = st[0] <= st[1] ? 0 : 1;
        const int out = 1 - in;
        if (st[in] < K) return BSA_ERR_SHAPE;
        if (st[out] < (n[in] - 1) * st[in] + K) return BSA_ERR_SHAPE;
    }
    return BSA_OK;
}

// BSA_SELECT_PATH=row|group|pair overrides the policy's choice among the
// paths that can serve a call (for benchmarking); -1 when unset.
int forced_path() {
    static const int v = [] {
        const char* e = getenv("BSA_SELECT_PATH");
        if (e == nullptr) return -1;
        if (strcmp(e, "row") == 0) return BSA_PATH_ROW;
        if (strcmp(e, "group") == 0) return BSA_PATH_GROUP;
        if (strcmp(e, "pair") == 0) return BSA_PATH_PAIR;
        if (strcmp(e, "octet") == 0) return BSA_PATH_OCTET;
        if (strcmp(e, "wide") == 0) return BSA_PATH_WIDE;
        return -1;
    }();
    return v;
}

// The launch policy (see bsa_select_policy in the header).
int make_policy(int64_t rows, int64_t M, int32_t K, int32_t dtype, int32_t num_sms,
                bsa_launch_policy_t* p) {
    memset(p, 0, sizeof(*p));
    const int vec = dtype == BSA_DTYPE_BF16 ? 8 : 4;
    // Vectors per lane per pass: smallest of 1, 2, 4 covering the capacity.
    int nv = 4;
    if (M <= 32LL * 1 * vec) nv = 1;
    else if (M <= 32LL * 2 * vec) nv = 2;
    const int64_t per_pass = 32LL * nv * vec;
    const int64_t passes = (M + per_pass - 1) / per_pass;
    // Representatives for the threshold estimate: enough for K' <= K.
    int reps = 2 * nv;
    if (K <= 16) reps = 1;
    else if (K <= 48) reps = 2;
    // Split a long row over several warps only when rows alone cannot
    // occupy the GPU (about 32 resident warps per SM).
    const int64_t resident = (int64_t)num_sms * 32;
    int64_t chunks = 1;
    if (passes > 1 && rows < resident) {
        chunks = resident / (rows > 0 ? rows : 1);
        if (chunks > passes) chunks = passes;
        if (chunks < 1) chunks = 1;
    }
    int warps = 8;
    const int cap = (int)((K + 32 * vec + 31) / 32 * 32);
    int smem = warps * cap * 8;
    // Pair path (2 lanes per row, 16 rows per warp) for topk <= 32 and rows
    // of at most 2 KB; the group path (4 lanes per row) is kept selectable for
    // comparison.  Both fall back to the warp path for overflowing rows.
    const int elem = dtype == BSA_DTYPE_BF16 ? 2 : 4;
    const int forced = forced_path();
    const bool short_rows = M * elem <= kGroupMaxBytes;
    // buffers wider than 2 KB whose rows are not split: the pair and octet
    // paths take the rows whose range fits in 2 KB and list the others for a
    // second, wide-path launch
    const bool tail = !short_rows && chunks == 1 && cap <= kWideMaxCap;
    const bool pair_ok = K <= kGroupMaxK && (short_rows || tail);
    const bool oct_ok = K <= kOctMaxK && (short_rows || tail);
    const int32_t long_grid = tail ? num_sms * kWideCtasPerSm : 0;
    // Wide path alone (one warp per row, every row), for calls with topk <=
    // 64, when forced.
    const bool wide_ok = K <= kOctMaxK && cap <= kWideMaxCap;
    if (wide_ok && forced == BSA_PATH_WIDE) {
        int64_t grid = (rows + kWideWarps - 1) / kWideWarps;
        if (grid > INT32_MAX) grid = INT32_MAX;
        if (grid < 1) grid = 1;
        p->path = BSA_PATH_WIDE;
        p->vecs_per_lane = 4;
        p->chunks_per_row = 1;
        p->reps_per_lane = 16;
        p->warps_per_cta = kWideWarps;
        p->grid = (int32_t)grid;
        p->cand_capacity = cap;
        p->smem_bytes = kWideWarps * (int)sizeof(WideSmem);
        return BSA_OK;
    }
    // Octet path (8 lanes per row, 4 rows per warp) for 32 < topk <= 64, or
    // for any topk <= 64 when forced.
    if (oct_ok && (forced == BSA_PATH_OCTET || (!pair_ok && forced != BSA_PATH_ROW))) {
        const int64_t items = (rows + kOctRows - 1) / kOctRows;
        int64_t grid = (items + kOctWarps - 1) / kOctWarps;
        if (grid > INT32_MAX) grid = INT32_MAX;
        if (grid < 1) grid = 1;
        p->path = BSA_PATH_OCTET;
        p->vecs_per_lane = 4;
        p->chunks_per_row = 1;
        p->reps_per_lane = 16;
        p->warps_per_cta = kOctWarps;
        p->grid = (int32_t)grid;
        p->cand_capacity = cap;
        p->smem_bytes = kOctWarps * (int)sizeof(OctSmem);
        p->long_rows = tail ? 1 : 0;
        p->long_grid = long_grid;
        return BSA_OK;
    }
    if (pair_ok && forced != BSA_PATH_ROW && forced != BSA_PATH_GROUP) {
        const int gsmem = kPairWarps * (int)(dtype == BSA_DTYPE_BF16
                                                 ? sizeof(PairSmem<uint32_t>)
                                                 : sizeof(PairSmem<unsigned long long>));
        // One item (16 rows) per warp and no persistent grid: the hardware
        // hands a finished CTA's slot to the next CTA, which balances items
        // of unequal length better than a fixed stride over resident warps.
        // (The kernel still strides, so a capped grid would also be correct.)
        const int64_t items = (rows + kPairRows - 1) / kPairRows;
        int64_t grid = (items + kPairWarps - 1) / kPairWarps;
        if (grid > INT32_MAX) grid = INT32_MAX;
        if (grid < 1) grid = 1;
        p->path = BSA_PATH_PAIR;
        p->vecs_per_lane = 4;
        p->chunks_per_row = 1;
        p->reps_per_lane = 16;
        p->warps_per_cta = kPairWarps;
        p->grid = (int32_t)grid;
        p->cand_capacity = cap;
        p->smem_bytes = gsmem;
        p->long_rows = tail ? 1 : 0;
        p->long_grid = long_grid;
        return BSA_OK;
    }
    if (K <= kGroupMaxK && M * elem <= kGroupMaxBytes && forced != BSA_PATH_ROW) {
        const int gsmem = warps * (int)(dtype == BSA_DTYPE_BF16
                                            ? sizeof(GroupSmem<uint32_t>)
                                            : sizeof(GroupSmem<unsigned long long>));
        int ctas = 3;
        while (ctas > 1 && ctas * (gsmem + 1024) > 228 * 1024) --ctas;
        const int64_t items = (rows + kGroupRows - 1) / kGroupRows;
        int64_t grid = (items + warps - 1) / warps;
        const int64_t grid_cap = (int64_t)num_sms * ctas;
        if (grid > grid_cap) grid = grid_cap;
        if (grid < 1) grid = 1;
        p->path = BSA_PATH_GROUP;
        p->vecs_per_lane = 4;
        p->chunks_per_row = 1;
        p->reps_per_lane = 8;
        p->warps_per_cta = warps;
        p->grid = (int32_t)grid;
        p->cand_capacity = cap;
        p->smem_bytes = gsmem;
        return BSA_OK;
    }
    // One work item per warp; the grid is not capped at the resident CTAs,
    // so the hardware balances items of unequal length (the kernel strides,
    // so any grid is correct).
    const int64_t items = rows * chunks;
    int64_t grid = (items + warps - 1) / warps;
    if (grid > INT32_MAX) grid = INT32_MAX;
    if (grid < 1) grid = 1;
    p->path = chunks > 1 ? BSA_PATH_SPLIT : BSA_PATH_ROW;
    p->vecs_per_lane = nv;
    p->chunks_per_row = (int32_t)chunks;
    p->reps_per_lane = reps;
    p->warps_per_cta = warps;
    p->grid = (int32_t)grid;
    p->cand_capacity = cap;
    p->smem_bytes = smem;
    return BSA_OK;
}

int run_select(SelectArgs& a, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    bsa_launch_policy_t pol;
    const int64_t rows = a.T * a.H;
    if (rows > INT32_MAX) return BSA_ERR_SHAPE;
    make_policy(rows, a.M, a.K, a.dtype, device_sm_count(), &pol);
    const size_t need = select_workspace_bytes(rows, pol, a.K);
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes < need ||
            (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
            return BSA_ERR_WORKSPACE;
    }
    if (pol.long_rows) {
        SplitWorkspace ws{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
        ws.long_list = static_cast<int32_t*>(workspace);
        ws.long_count = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) +
                                                    align_up((size_t)rows * 4));
        // the list starts empty and untaken on every call (one memset node
        // in a graph)
        cudaError_t e = cudaMemsetAsync(ws.long_count, 0, 2 * sizeof(uint32_t), stream);
        if (e != cudaSuccess) return (int)e;
        return status_of(launch_select(a, pol, ws, stream));
    }
    SplitWorkspace ws = carve_split_workspace(workspace, rows, pol.chunks_per_row, a.K);
    if (need > 0) {
        // The merge tickets start at zero on every call, whatever an earlier
        // call with another layout left in this memory (one memset node when
        // captured in a graph).
        cudaError_t e = cudaMemsetAsync(ws.tickets, 0, (size_t)rows * sizeof(int32_t), stream);
        if (e != cudaSuccess) return (int)e;
    }
    return status_of(launch_select(a, pol, ws, stream));
}

}  // namespace

extern "C" {

const char* bsa_status_string(int status) {
    switch (status) {
        case BSA_OK: return "ok";
        case BSA_ERR_NULL: return "a required pointer is NULL";
        case BSA_ERR_SHAPE: return "invalid size or stride";
        case BSA_ERR_TOPK: return "invalid topk / num_init / num_local";
        case BSA_ERR_DTYPE: return "unknown score dtype";
        case BSA_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        case BSA_ERR_ROWS: return "T != num_reqs * decode_query_len";
        case BSA_ERR_ALIGN: return "scores pointer not aligned to its element size";
        case BSA_ERR_CAPACITY: return "request needs more scratch than the built-in array holds";
        default: break;
    }
    if (status > 0) return cudaGetErrorString((cudaError_t)status);
    return "unknown status";
}

int bsa_select_policy(int64_t rows, int64_t M, int32_t K, int32_t dtype, int32_t num_sms,
                      bsa_launch_policy_t* policy) {
    if (policy == nullptr) return BSA_ERR_NULL;
    if (dtype != BSA_DTYPE_BF16 && dtype != BSA_DTYPE_FP32) return BSA_ERR_DTYPE;
    if (rows < 0 || M < 1 || M > BSA_MAX_K_TILES || num_sms < 1) return BSA_ERR_SHAPE;
    if (K < 1 || K > BSA_MAX_TOPK || K > M) return BSA_ERR_TOPK;
    return make_policy(rows, M, K, dtype, num_sms, policy);
}

size_t bsa_topk_workspace_bytes(int64_t T, int64_t H, int64_t M, int32_t K, int32_t dtype) {
    if (T <= 0 || H <= 0 || M < 1 || M > BSA_MAX_K_TILES || K < 1 || K > BSA_MAX_TOPK || K > M)
        return 0;
    if (dtype != BSA_DTYPE_BF16 && dtype != BSA_DTYPE_FP32) return 0;
    bsa_launch_policy_t pol;
    make_policy(T * H, M, K, dtype, device_sm_count(), &pol);
    return select_workspace_bytes(T * H, pol, K);
}

int bsa_num_valid_pages_decode(const int32_t* seq_lens, int64_t num_reqs, int32_t dql,
                               int32_t* num_valid_pages, void* stream) {
    if (num_reqs < 0 || dql < 1) return BSA_ERR_SHAPE;
    if (num_reqs == 0) return BSA_OK;
    if (seq_lens == nullptr || num_valid_pages == nullptr) return BSA_ERR_NULL;
    return status_of(launch_num_valid_pages_decode(seq_lens, num_reqs, dql, num_valid_pages,
                                                   static_cast<cudaStream_t>(stream)));
}

int bsa_num_valid_pages_varlen(const int32_t* cu_seqlens_q, const int32_t* prefix_lens,
                               int64_t num_seqs, int64_t total_q, int32_t* num_valid_pages,
                               void* stream) {
    if (num_seqs < 0 || total_q < 0) return BSA_ERR_SHAPE;
    if (total_q == 0) return BSA_OK;
    if (num_valid_pages == nullptr || cu_seqlens_q == nullptr ||
        (num_seqs > 0 && prefix_lens == nullptr))
        return BSA_ERR_NULL;
    return status_of(launch_num_valid_pages_varlen(cu_seqlens_q, prefix_lens, num_seqs, total_q,
                                                   num_valid_pages,
                                                   static_cast<cudaStream_t>(stream)));
}

int bsa_topk_select(const void* scores, int32_t dtype, int64_t T, int64_t H, int64_t M,
                    int64_t token_stride, int64_t head_stride, const int32_t* num_valid_pages,
                    int32_t K, int32_t num_init, int32_t num_local, int32_t* out_idx,
                    int64_t out_token_stride, int64_t out_head_stride, void* workspace,
                    size_t workspace_bytes, void* stream) {
    if (dtype != BSA_DTYPE_BF16 && dtype != BSA_DTYPE_FP32) return BSA_ERR_DTYPE;
    if (T < 0 || H < 0 || M < 1 || M > BSA_MAX_K_TILES) return BSA_ERR_SHAPE;
    int rc = check_topk_args(M, K, num_init, num_local);
    if (rc != BSA_OK) return rc;
    if (head_stride < M || token_stride < (H > 0 ? (H - 1) * head_stride + M : M))
        return BSA_ERR_SHAPE;
    rc = check_out_layout(T, H, K, out_token_stride, out_head_stride);
    if (rc != BSA_OK) return rc;
    if (T == 0 || H == 0) return BSA_OK;
    if (scores == nullptr || num_valid_pages == nullptr || out_idx == nullptr) return BSA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(scores) % elem_bytes(dtype)) != 0) return BSA_ERR_ALIGN;
    SelectArgs a{};
    a.scores = scores;
    a.dtype = dtype;
    a.T = T;
    a.H = H;
    a.M = M;
    a.token_stride = token_stride;
    a.head_stride = head_stride;
    a.num_valid_pages = num_valid_pages;
    a.dql = 1;
    a.K = K;
    a.num_init = num_init;
    a.num_local = num_local;
    a.out_idx = out_idx;
    a.out_ts = out_token_stride;
    a.out_hs = out_head_stride;
    a.fused = false;
    a.table = false;
    return run_select(a, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int bsa_build_sparse_block_table(const int32_t* topk_idx, int64_t T, int64_t H, int32_t K,
                                 const int32_t* block_table, int64_t num_reqs,
                                 int64_t max_blocks, const int32_t* seq_lens,
                                 int32_t decode_query_len, int32_t* sparse_bt,
                                 int32_t* sparse_ctx, void* stream) {
    if (T < 0 || H < 0 || num_reqs < 0 || max_blocks < 0 || decode_query_len < 1)
        return BSA_ERR_SHAPE;
    if (K < 1 || K > BSA_MAX_TOPK) return BSA_ERR_TOPK;
    if (T != num_reqs * decode_query_len) return BSA_ERR_ROWS;
    if (T == 0 || H == 0) return BSA_OK;
    if (topk_idx == nullptr || seq_lens == nullptr || sparse_bt == nullptr ||
        sparse_ctx == nullptr || (max_blocks > 0 && block_table == nullptr))
        return BSA_ERR_NULL;
    return status_of(launch_build_sparse_block_table(topk_idx, T, H, K, block_table, max_blocks,
                                                     seq_lens, decode_query_len, sparse_bt,
                                                     sparse_ctx,
                                                     static_cast<cudaStream_t>(stream)));
}

int bsa_topk_select_sparse_table(const void* scores, int32_t dtype, int64_t num_reqs,
                                 int32_t decode_query_len, int64_t H, int64_t M,
                                 int64_t token_stride, int64_t head_stride,
                                 const int32_t* seq_lens, int32_t K, int32_t num_init,
                                 int32_t num_local, const int32_t* block_table,
                                 int64_t max_blocks, int32_t* out_idx,
                                 int64_t out_token_stride, int64_t out_head_stride,
                                 int32_t* sparse_bt, int32_t* sparse_ctx, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    if (dtype != BSA_DTYPE_BF16 && dtype != BSA_DTYPE_FP32) return BSA_ERR_DTYPE;
    if (num_reqs < 0 || decode_query_len < 1 || H < 0 || M < 1 || M > BSA_MAX_K_TILES ||
        max_blocks < 0)
        return BSA_ERR_SHAPE;
    int rc = check_topk_args(M, K, num_init, num_local);
    if (rc != BSA_OK) return rc;
    if (head_stride < M || token_stride < (H > 0 ? (H - 1) * head_stride + M : M))
        return BSA_ERR_SHAPE;
    const int64_t T = num_reqs * decode_query_len;
    if (out_idx != nullptr) {
        rc = check_out_layout(T, H, K, out_token_stride, out_head_stride);
        if (rc != BSA_OK) return rc;
    }
    if (T == 0 || H == 0) return BSA_OK;
    if (scores == nullptr || seq_lens == nullptr || sparse_bt == nullptr ||
        sparse_ctx == nullptr || (max_blocks > 0 && block_table == nullptr))
        return BSA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(scores) % elem_bytes(dtype)) != 0) return BSA_ERR_ALIGN;
    SelectArgs a{};
    a.scores = scores;
    a.dtype = dtype;
    a.T = T;
    a.H = H;
    a.M = M;
    a.token_stride = token_stride;
    a.head_stride = head_stride;
    a.seq_lens = seq_lens;
    a.dql = decode_query_len;
    a.K = K;
    a.num_init = num_init;
    a.num_local = num_local;
    a.out_idx = out_idx;
    a.out_ts = out_token_stride;
    a.out_hs = out_head_stride;
    a.block_table = block_table;
    a.max_blocks = max_blocks;
    a.sparse_bt = sparse_bt;
    a.sparse_ctx = sparse_ctx;
    a.fused = true;
    a.table = true;
    return run_select(a, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int bsa_index_score_topk_select(const void* q_idx, const void* k_idx, int64_t num_phys_blocks,
                                int64_t H, int64_t D, const int32_t* block_table,
                                int64_t max_blocks, const int32_t* seq_lens, int64_t num_reqs,
                                int32_t decode_query_len, float* scores, int64_t M,
                                int64_t token_stride, int64_t head_stride, int32_t K,
                                int32_t num_init, int32_t num_local, int32_t* out_idx,
                                int64_t out_token_stride, int64_t out_head_stride,
                                int32_t* sparse_bt, int32_t* sparse_ctx, void* stream) {
    if (num_reqs < 0 || decode_query_len < 1 || H < 1 || M < 1 || M > BSA_MAX_K_TILES ||
        max_blocks < 0 || num_phys_blocks < 0)
        return BSA_ERR_SHAPE;
    if (D < 8 || D > BSA_MAX_INDEX_DIM || D % 8 != 0) return BSA_ERR_SHAPE;
    if ((int64_t)decode_query_len * H > BSA_MAX_INDEX_QUERIES) return BSA_ERR_SHAPE;
    int rc = check_topk_args(M, K, num_init, num_local);
    if (rc != BSA_OK) return rc;
    if (head_stride < M || token_stride < (H - 1) * head_stride + M) return BSA_ERR_SHAPE;
    const int64_t T = num_reqs * decode_query_len;
    rc = check_out_layout(T, H, K, out_token_stride, out_head_stride);
    if (rc != BSA_OK) return rc;
    if ((sparse_bt == nullptr) != (sparse_ctx == nullptr)) return BSA_ERR_NULL;
    if (T == 0) return BSA_OK;
    if (q_idx == nullptr || k_idx == nullptr || seq_lens == nullptr || scores == nullptr ||
        out_idx == nullptr || (max_blocks > 0 && block_table == nullptr))
        return BSA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(q_idx) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(k_idx) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(scores) & 3) != 0)
        return BSA_ERR_ALIGN;
    SelectArgs a{};
    a.scores = scores;
    a.dtype = BSA_DTYPE_FP32;
    a.T = T;
    a.H = H;
    a.M = M;
    a.token_stride = token_stride;
    a.head_stride = head_stride;
    a.seq_lens = seq_lens;
    a.dql = decode_query_len;
    a.K = K;
    a.num_init = num_init;
    a.num_local = num_local;
    a.out_idx = out_idx;
    a.out_ts = out_token_stride;
    a.out_hs = out_head_stride;
    a.block_table = block_table;
    a.max_blocks = max_blocks;
    a.sparse_bt = sparse_bt;
    a.sparse_ctx = sparse_ctx;
    a.fused = true;
    a.table = sparse_bt != nullptr;
    return status_of(launch_index_score_select(a, static_cast<const uint16_t*>(q_idx),
                                               static_cast<const uint16_t*>(k_idx),
                                               num_phys_blocks, (int32_t)D, scores,
                                               static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

extern "C" int bsa_set_status_word(uint32_t* word) {
    if ((reinterpret_cast<uintptr_t>(word) & 3) != 0) return BSA_ERR_ALIGN;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return BSA_ERR_SHAPE;
    g_status_word[dev].store(word, std::memory_order_release);
    return BSA_OK;
}

extern "C" int bsa_read_status(uint32_t* out, int32_t clear, void* stream) {
    if (out == nullptr) return BSA_ERR_NULL;
    *out = 0;
    uint32_t* word = current_status_word();
    if (word == nullptr) return BSA_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t got = 0;
    cudaError_t e = cudaMemcpyAsync(&got, word, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(word, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return (int)e;
    *out = got;
    return BSA_OK;
}
