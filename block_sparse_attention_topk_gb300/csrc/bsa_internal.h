// bsa_internal.h -- declarations shared by the library's translation units
// (host launchers and the launch policy).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/bsa_topk.h"

namespace bsa {

constexpr int kPageSize = BSA_PAGE_SIZE;              // tokens per sparse block
constexpr int kSubPage = BSA_SUB_PAGE_SIZE;           // tokens per table entry
constexpr int kPagesPerBlock = BSA_PAGES_PER_SPARSE_BLOCK;
constexpr int kLogPageSize = 7;

// Group path: 4 lanes per row, 8 rows per warp (see bsa_select.cu).
constexpr int kGroupLanes = 4;       // lanes per row
constexpr int kGroupRows = 8;        // rows per warp
constexpr int kGroupMaxVecs = 130;   // 16-byte vectors per row the group path covers
constexpr int kGroupCand = 32;       // candidate capacity per row (one 4-lane sort)
constexpr int kGroupMaxK = 32;       // largest topk the group path serves
constexpr int kGroupMaxBytes = 2048; // capacity x element size the group path covers
constexpr int kGroupStepsPad = 40;   // >= ceil(kGroupMaxVecs / kGroupLanes), multiple of 8

struct GroupRowDesc {
    unsigned long long v0;       // first 16-byte vector of the non-forced range
    unsigned long long row_ptr;  // address of element 0 of the row
    int32_t base_id, lo, hi, theta;
    int32_t fast, nvec;
};

// Shared memory of one warp of the group path.  CK is the composite key type
// (uint32 for bf16, uint64 for fp32).
template <typename CK>
struct GroupSmem {
    // per-vector maxima (raw signed), lane-major: vector k = q + 4 i of row g
    // at vmax[g][q][i]
    int16_t vmax[kGroupRows][kGroupLanes][kGroupStepsPad];
    union {
        uint16_t queue[kGroupRows * kGroupMaxVecs];  // (row << 13 | vector) work items
        struct {
            int32_t sorted[kGroupRows][kGroupMaxK];  // selected ids, ascending
        } s;
    } q;
    CK cand[kGroupRows][kGroupCand];           // candidate composite keys
    int32_t ccount[kGroupRows];
    int32_t ovf[kGroupRows];
    GroupRowDesc desc[kGroupRows];
};

// Pair path: 2 lanes per row, 16 rows per warp, 32-byte chunks (see bsa_select.cu).
constexpr int kPairRows = 16;        // rows per warp
constexpr int kPairMaxChunks = 66;   // 32-byte chunks per row (2 KB + alignment)
constexpr int kPairStepsPad = 40;    // >= ceil(kPairMaxChunks / 2), multiple of 8
constexpr int kPairCand = 32;        // candidate capacity per row (one 2-lane sort)
constexpr int kPairWarps = 4;        // warps per CTA
constexpr int kPairCtas = 5;         // CTAs per SM the fused kernel's register bound allows
constexpr int kPairCtasSelect = 6;   // the same for the plain bf16 select (no table epilogue)

struct PairRowDesc {
    unsigned long long c0;       // first 32-byte chunk of the non-forced range
    unsigned long long row_ptr;  // address of element 0 of the row
    int32_t base_id, lo, hi, theta;
    int32_t nchunk;
    int32_t inside;              // every chunk of the range lies inside the score buffer
};

template <typename CK>
struct PairSmem {
    union {
        // chunk maxima (signed keys; fp32 keeps the top 16 bits): the two
        // chunks 4 i + 2 s + c (c = 0, 1) a lane takes at step i share one
        // word, vmax2[i][lane] = max(c = 0) | max(c = 1) << 16; live from
        // pass 1 until the queue is built
        uint32_t vmax2[kPairStepsPad / 2][32];
        // one 32-byte chunk per lane while candidates are collected
        uint32_t scratch[32][8];
    } a;
    union {
        uint16_t queue[kPairRows * kPairMaxChunks];  // (row << 8 | chunk) work items
        int32_t sorted[kPairRows][kGroupMaxK];      // selected ids, ascending
    } q;
    CK cand[kPairRows][kPairCand];                  // candidate composite keys
    int32_t ccount[kPairRows];
    int32_t ovf[kPairRows];
    PairRowDesc desc[kPairRows];
};

// Octet path: 8 lanes per row, 4 rows per warp, for 32 < topk <= 64 (see
// bsa_select.cu).
constexpr int kOctLanes = 8;         // lanes per row
constexpr int kOctRows = 4;          // rows per warp
constexpr int kOctCand = 128;        // candidate capacity per row (16 per lane)
constexpr int kOctMaxK = 64;         // largest topk the octet path serves
constexpr int kOctWarps = 4;         // warps per CTA
constexpr int kOctCtas = 6;          // CTAs per SM of the fused kernel (register bound)
constexpr int kOctCtasSelect = 7;    // the same for the plain bf16 select

struct OctSmem {
    union {
        int32_t ckey[kOctRows][kOctCand];     // candidate keys (signed order-preserving), id order
        int16_t ckey16[kOctRows][kOctCand];   // the same for bf16
    };
    uint16_t cid[kOctRows][kOctCand];   // their block ids
    int32_t sorted[kOctRows][kOctMaxK]; // selected non-forced ids, ascending
    uint32_t scratch[32][8];            // one 32-byte chunk per lane while candidates are read out
};

// Wide path: one warp per row, for rows longer than 2 KB and topk <= 64 (see
// bsa_select.cu).
constexpr int kWideCand = 256;       // candidate capacity per row (8 per lane)
constexpr int kWideWarps = 4;        // warps per CTA, one row each
constexpr int kWideMaxCap = 320;     // warp-path buffer entries an overflowing row needs (topk <= 64)
constexpr int kWideCtasPerSm = 6;    // resident CTAs per SM (register bound), for persistent grids
constexpr int kWideHotChunks = 1024; // rows of up to 32 KB keep their chunk maxima for pass 2

struct WideSmem {
    union {
        struct {
            union {
                int16_t ckey[kWideCand];    // candidate keys (signed order-preserving), id order: bf16
                int32_t ckey32[kWideCand];  // the same for fp32
            };
            uint16_t cid[kWideCand];      // their block ids
            int32_t sorted[kOctMaxK];     // selected non-forced ids, ascending
        } c;
        uint32_t fallback[2 * kWideMaxCap];  // the warp path's keys and ids
    };
    uint32_t scratch[32][8];              // one 32-byte chunk per lane while candidates are read out
    int16_t cmax[kWideHotChunks];         // each interior chunk's maximum (pass 1): bf16 raw, fp32 key's top 16 bits
    uint16_t hot[kWideHotChunks];         // the chunks pass 2 reads, ascending
};

// Everything one selector launch needs.  Pointers are device pointers.
struct SelectArgs {
    const void* scores;
    int32_t dtype;
    int64_t T, H, M;
    int64_t token_stride, head_stride;
    const int32_t* num_valid_pages;   // select mode: int32[T]
    const int32_t* seq_lens;          // fused mode: int32[T / dql]
    int32_t dql;
    int32_t K, num_init, num_local;
    int32_t* out_idx;                 // may be null in fused mode
    int64_t out_ts, out_hs;           // element strides of out_idx rows (token, head)
    const int32_t* block_table;       // fused mode
    int64_t max_blocks;
    int32_t* sparse_bt;
    int32_t* sparse_ctx;
    bool fused;                       // rows are decode rows: page counts from seq_lens
    bool table;                       // the sparse-table epilogue is written
    uint32_t* status;                 // the device status word, or null (no checks)
    // x / H and x / dql for x < 2^31 as (umulhi(x, mul) + x) >> shift
    uint32_t h_mul, h_shift, dql_mul, dql_shift;
};

#ifdef __CUDACC__
// Sets `bit` in the status word when `bad` holds and a word is registered.
__device__ __forceinline__ void report_status(uint32_t* word, bool bad, uint32_t bit) {
    if (word != nullptr && bad) atomicOr(word, bit);
}
// A physical block id whose page ids phys * 8 + p are not valid int32 page ids.
__device__ __forceinline__ bool bad_phys_block(int32_t phys) {
    return (uint32_t)phys > (uint32_t)BSA_MAX_PHYS_BLOCK;
}

// One 256-bit store of eight int32 (a full 32-byte sector); p 32-byte aligned.
__device__ __forceinline__ void st_v8(int32_t* p, const int32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
#endif

// Multiplier and shift that divide every x < 2^31 by d >= 1 exactly as
// (umulhi(x, mul) + x) >> shift (round-up reciprocal, Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994).
inline void div_magic(uint32_t d, uint32_t* mul, uint32_t* shift) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    *mul = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
    *shift = l;
}

// Workspace carve-up for the split path (all offsets 256-byte aligned).
struct SplitWorkspace {
    uint32_t* keys;     // [rows, chunks, K]
    int32_t* ids;       // [rows, chunks, K]
    int32_t* counts;    // [rows, chunks]
    int32_t* tickets;   // [rows]
    // pair / octet paths with long_rows: the rows left to the wide path
    int32_t* long_list;     // [rows]
    uint32_t* long_count;   // [0]: entries in long_list, [1]: entries past the first grid stride taken (zeroed per call)
};

size_t split_workspace_bytes(int64_t rows, int32_t chunks, int32_t K);
SplitWorkspace carve_split_workspace(void* base, int64_t rows, int32_t chunks, int32_t K);

int device_sm_count();

// The status word registered for the current device (bsa_set_status_word), or null.
uint32_t* current_status_word();

// Launches the selector (plain or fused) with a policy from bsa_select_policy.
cudaError_t launch_select(const SelectArgs& a, const bsa_launch_policy_t& pol,
                          const SplitWorkspace& ws, cudaStream_t stream);

// Fused index score + select of decode rows (see bsa_select.cu); `a` holds
// the selection over the fp32 score buffer `scores`.
cudaError_t launch_index_score_select(const SelectArgs& a, const uint16_t* q, const uint16_t* k,
                                      int64_t nb, int32_t D, float* scores, cudaStream_t stream);

cudaError_t launch_num_valid_pages_decode(const int32_t* seq_lens, int64_t num_reqs,
                                          int32_t dql, int32_t* out, cudaStream_t stream);
cudaError_t launch_num_valid_pages_varlen(const int32_t* cu, const int32_t* prefix,
                                          int64_t num_seqs, int64_t total_q, int32_t* out,
                                          cudaStream_t stream);
cudaError_t launch_build_sparse_block_table(const int32_t* topk_idx, int64_t T, int64_t H,
                                            int32_t K, const int32_t* block_table,
                                            int64_t max_blocks, const int32_t* seq_lens,
                                            int32_t dql, int32_t* sparse_bt,
                                            int32_t* sparse_ctx, cudaStream_t stream);

}  // namespace bsa
