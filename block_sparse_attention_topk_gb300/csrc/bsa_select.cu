// bsa_select.cu -- the top-k block selector (plain and fused with the sparse
// block table) for GB300 / sm_103a.
//
// What it computes (vLLM PR #47502 report, "[Minimax-M3] Using
// tok_sparse_select from MSA instead of triton kernels", sections 实现拆解 and
// 关键源码片段, indexer_msa.py):
// for every row (token t, index head h) of the unified token-major score
// buffer, the top-K block ids among the causal prefix b < v = min(M,
// num_valid_pages[t]), with the init blocks [0, I) and the local blocks
// [v - L, v) always kept.  Scores are ordered by IEEE totalOrder, ties go to
// the lower block id (vLLM PR #55235 report, sections 执行摘要 and 评论区精华:
// NaN, +-Inf, +-0 and tied scores each have a fixed place).  The fused variant
// adds the page-16 sparse block-table epilogue of vLLM PR #47984 report
// ("Support speculative decode with AITER sparse PA", 实现拆解 items 1 and 3)
// and of the EMIT_SPARSE_TABLE flag in PR #55235.
//
// How (a design for this GPU, not the pages' Triton/ROCm kernels).  The
// selector kernels share one method:
//  * Threshold.  Representatives (maxima of disjoint element subsets) give a
//    lower bound theta on the K'-th best non-forced score: K' distinct
//    elements reach the K'-th largest representative.  Only elements >= theta
//    can be selected; for N(0,1)-like scores that is about K' to 1.5 K'.
//    Forced blocks (init [0, I), local [v - L, v)) and ids outside the causal
//    prefix are masked out of the search and emitted directly.
//  * Candidates are composite keys (order-preserving key, then the inverted
//    id): unique, and larger means a better (score, lower id) pair.  An exact
//    select keeps the K' largest; the output lists init ids, the selected ids
//    and local ids in ascending order, then -1.
//  * pair_select_kernel (default for topk <= 32 and rows <= 2 KB): 2 lanes per
//    row, 16 rows per warp, 32-byte chunks; elements become signed
//    order-preserving keys as they are loaded (IEEE totalOrder for any sign);
//    chunk maxima select the hot chunks, which are reloaded (L2 hits) and
//    filtered; bitonic networks across the lane pair sort representatives and
//    candidates.  Rows whose candidates overflow are redone by the warp path.
//  * octet_select_kernel (default for 32 < topk <= 64 and rows <= 2 KB): 8
//    lanes per row, 4 rows per warp; position maxima as representatives,
//    packed sorting networks for theta, an id-ordered candidate list and an
//    exact kappa search.
//  * wide_select_kernel (rows over 2 KB, topk <= 64): the octet method
//    with all 32 lanes on one row, and a list of the chunks that reach
//    theta.  On a buffer wider than 2 KB (the 8192-tile capture-time
//    capacity) the pair and octet kernels take every row whose range fits in
//    2 KB and list the others, which a second launch takes with this kernel.
//  * group_select_kernel: the pair method with 4 lanes per row, 8 rows per
//    warp (selectable for testing).
//  * select_kernel (warp path): one warp per row, or per chunk of a long row
//    when there are too few rows to fill the GPU (split path).  Candidates
//    are appended in id order to a per-warp shared buffer compacted by an
//    exact warp select (bit search over the key, ties by buffer order).  A
//    split row's chunks write their lists to the caller's workspace and take a
//    ticket with atomicAdd; the last arriver merges, writes the output and
//    resets the ticket, and the host clears the tickets before every launch
//    (PR #55235: counters reset under graph replay).  Nothing waits on another
//    warp.
//  * The fused variant of every kernel gathers block_table[req, b] for the
//    selected blocks and writes their page-16 entries and ctx in the same pass.
//  * index_score_select_kernel (further down) computes decode index scores
//    into the unified buffer and selects from them in the same launch.
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kWarpsPerCta = 8;
constexpr int kThreads = kWarpsPerCta * 32;

__device__ __forceinline__ uint32_t max_s16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t min_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t min_s16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("min.s16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// The same through L2 only (coherent with writes made earlier in the kernel,
// which the non-coherent path above is not).
__device__ __forceinline__ uint4 ld_cg_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// ---------------------------------------------------------------------------
// Element types.  `raw` is the bit pattern sign-extended to int32; `key` is
// the order-preserving unsigned key: larger key <=> later in totalOrder.
// ---------------------------------------------------------------------------
template <bool BF16>
struct Elem;

template <>
struct Elem<true> {
    static constexpr int kVec = 8;                 // elements per 16 bytes
    static constexpr int kBytes = 2;
    static constexpr int kKeyBits = 16;
    static constexpr uint32_t kKeyMax = 0xFFFFu;
    static constexpr uint32_t kKeyOfPlusZero = 0x8000u;
    static constexpr uint32_t kMaskWord = 0x80008000u;
    static constexpr int kThetaTop = 14, kThetaLow = 0;  // bits searched for theta
    __device__ static int32_t raw(const uint4& w, int e) {
        uint32_t word = e < 2 ? w.x : e < 4 ? w.y : e < 6 ? w.z : w.w;
        return (int32_t)(int16_t)(uint16_t)(word >> ((e & 1) * 16));
    }
    __device__ static uint32_t key(int32_t raw) {
        uint32_t u = (uint32_t)raw & 0xFFFFu;
        return (u & 0x8000u) ? (~u & 0xFFFFu) : (u | 0x8000u);
    }
    __device__ static int32_t raw_of_nonneg_key(uint32_t k) { return (int32_t)(k - 0x8000u); }
    __device__ static int32_t load_one(const char* p) {
        return (int32_t)(int16_t)__ldg(reinterpret_cast<const unsigned short*>(p));
    }
    __device__ static int32_t load_one_cg(const char* p) {
        return (int32_t)(int16_t)__ldcg(reinterpret_cast<const unsigned short*>(p));
    }
    __device__ static void set(uint4& w, int e, int32_t raw) {
        uint32_t* word = e < 2 ? &w.x : e < 4 ? &w.y : e < 6 ? &w.z : &w.w;
        int sh = (e & 1) * 16;
        *word = (*word & ~(0xFFFFu << sh)) | (((uint32_t)raw & 0xFFFFu) << sh);
    }
    // Per-lane representatives: q = 0 / 1 are the two halves.
    __device__ static uint32_t slot_pack_max(const uint4& w) {
        return max_s16x2(max_s16x2(w.x, w.y), max_s16x2(w.z, w.w));
    }
    __device__ static int32_t pack_lo(uint32_t p) { return (int32_t)(int16_t)(uint16_t)p; }
    __device__ static int32_t pack_hi(uint32_t p) { return (int32_t)(int16_t)(uint16_t)(p >> 16); }
    // does any element of the packed maximum reach theta (theta >= 0)?
    __device__ static bool pack_any_ge(uint32_t p, int32_t theta) {
        return pack_lo(p) >= theta || pack_hi(p) >= theta;
    }
};

template <>
struct Elem<false> {
    static constexpr int kVec = 4;
    static constexpr int kBytes = 4;
    static constexpr int kKeyBits = 32;
    static constexpr uint32_t kKeyMax = 0xFFFFFFFFu;
    static constexpr uint32_t kKeyOfPlusZero = 0x80000000u;
    static constexpr uint32_t kMaskWord = 0x80000000u;
    static constexpr int kThetaTop = 30, kThetaLow = 16;  // bf16-resolution bound suffices
    __device__ static int32_t raw(const uint4& w, int e) {
        return (int32_t)(e == 0 ? w.x : e == 1 ? w.y : e == 2 ? w.z : w.w);
    }
    __device__ static uint32_t key(int32_t raw) {
        uint32_t u = (uint32_t)raw;
        return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    __device__ static int32_t raw_of_nonneg_key(uint32_t k) { return (int32_t)(k - 0x80000000u); }
    __device__ static int32_t load_one(const char* p) {
        return (int32_t)__ldg(reinterpret_cast<const unsigned int*>(p));
    }
    __device__ static int32_t load_one_cg(const char* p) {
        return (int32_t)__ldcg(reinterpret_cast<const unsigned int*>(p));
    }
    __device__ static void set(uint4& w, int e, int32_t raw) {
        uint32_t* word = e == 0 ? &w.x : e == 1 ? &w.y : e == 2 ? &w.z : &w.w;
        *word = (uint32_t)raw;
    }
    // "packed" maximum of a vector: (max of elements 0,2) | (max of 1,3) kept
    // as two int32 in a uint2-like pair; represented here as max over all for
    // q = 0 and the odd elements for q = 1 (see reps below).
    __device__ static int32_t even_max(const uint4& w) { return max((int32_t)w.x, (int32_t)w.z); }
    __device__ static int32_t odd_max(const uint4& w) { return max((int32_t)w.y, (int32_t)w.w); }
};

// ---------------------------------------------------------------------------
// Exact warp select on the shared candidate buffer: keep the `keep` best
// entries (key descending, buffer position ascending), preserving order.
// Returns the key of the worst kept entry.
// ---------------------------------------------------------------------------
template <int KEY_BITS>
__device__ uint32_t warp_compact(uint32_t* keys, int32_t* ids, int n, int keep, int lane) {
    const int rounds = (n + 31) >> 5;
    uint32_t kappa = 0;
    for (int bit = KEY_BITS - 1; bit >= 0; --bit) {
        const uint32_t t = kappa | (1u << bit);
        int c = 0;
        for (int s = 0; s < rounds; ++s) {
            const int e = (s << 5) + lane;
            c += (e < n && keys[e] >= t) ? 1 : 0;
        }
        c = __reduce_add_sync(kFull, c);
        if (c >= keep) kappa = t;
    }
    int above = 0;
    for (int s = 0; s < rounds; ++s) {
        const int e = (s << 5) + lane;
        above += (e < n && keys[e] > kappa) ? 1 : 0;
    }
    above = __reduce_add_sync(kFull, above);
    const int ties_wanted = keep - above;
    int ties_seen = 0, kept = 0;
    const unsigned lt = lanemask_lt();
    for (int s = 0; s < rounds; ++s) {
        const int e = (s << 5) + lane;
        const bool in = e < n;
        const uint32_t k = in ? keys[e] : 0u;
        const int32_t id = in ? ids[e] : 0;
        const bool gt = in && k > kappa;
        const bool eq = in && k == kappa;
        const unsigned eqb = __ballot_sync(kFull, eq);
        const bool take = gt || (eq && ties_seen + __popc(eqb & lt) < ties_wanted);
        ties_seen += __popc(eqb);
        const unsigned tb = __ballot_sync(kFull, take);
        const int pos = kept + __popc(tb & lt);
        __syncwarp();
        if (take) {
            keys[pos] = k;
            ids[pos] = id;
        }
        kept += __popc(tb);
        __syncwarp();
    }
    return kappa;
}

// Warp-wide exclusive prefix sum of `x`; `total` gets the sum.
__device__ __forceinline__ int warp_excl_scan(int x, int lane, int& total) {
    int incl = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += y;
    }
    total = __shfl_sync(kFull, incl, 31);
    return incl - x;
}

struct Split {
    uint32_t* keys;
    int32_t* ids;
    int32_t* counts;
    int32_t* tickets;
};

struct KernelParams {
    SelectArgs a;
    Split ws;
    int32_t* long_list;       // pair / octet paths: rows left to the wide path, or null
    uint32_t* long_count;     // [0]: entries in long_list; [1]: entries past the first grid stride taken
    int32_t chunks_per_row;   // work items per row
    int32_t vecs_per_chunk;   // vectors (16 B) per work item
    int32_t cap;              // candidate buffer entries per warp
    int64_t rows;
    uintptr_t buf_lo, buf_hi; // [first, last + 1) byte of the score buffer
};

// Candidate-buffer state of one warp.
struct Buf {
    uint32_t* keys;
    int32_t* ids;
    int n;            // entries held
    uint32_t kb;      // only keys >= kb can still be selected
    bool closed;      // nothing can enter any more (kept key is the maximum)
};

// Shrink the buffer to the `keep` best entries and raise the entry bound.
template <int KEY_BITS, uint32_t KEY_MAX>
__device__ __forceinline__ void buf_compact(Buf& b, int keep, int lane) {
    const uint32_t kappa = warp_compact<KEY_BITS>(b.keys, b.ids, b.n, keep, lane);
    b.n = keep;
    if (kappa == KEY_MAX) b.closed = true;
    else if (kappa + 1 > b.kb) b.kb = kappa + 1;
}

// Appends the candidates of one 32-lane group: lane holds `m` (bit i set =
// element i of its group is a candidate, keys/ids produced by `emit`).  The
// caller recomputes `m` after a compaction (the bound may have risen), so this
// returns false when it compacted and appended nothing.
template <int KEY_BITS, uint32_t KEY_MAX>
__device__ __forceinline__ bool buf_try_append(Buf& b, unsigned m, int cap, int keep, int lane,
                                               int& excl_out) {
    int total;
    const int excl = warp_excl_scan(__popc(m), lane, total);
    if (total == 0) {
        excl_out = -1;
        return true;
    }
    if (b.n + total > cap) {
        buf_compact<KEY_BITS, KEY_MAX>(b, keep, lane);
        return false;
    }
    excl_out = b.n + excl;
    b.n += total;
    return true;
}

// Output epilogue: ids, and in fused mode the page-16 table and ctx.
// sel(j): j < lo -> j (init); j - lo < kp -> buffered id; else hi + (j - lo - kp).
__device__ __forceinline__ int32_t selected_id(int j, int lo, int hi, int kp, bool all,
                                               const int32_t* buf_ids) {
    if (all || j < lo) return j;
    if (j - lo < kp) return buf_ids[j - lo];
    return hi + (j - lo - kp);
}

__device__ void write_outputs(const KernelParams& P, int64_t row, int64_t t, int64_t h, int n,
                              int lo, int hi, int kp, bool all, const int32_t* buf_ids,
                              int64_t causal_len, int64_t req, int lane) {
    const SelectArgs& a = P.a;
    const int K = a.K;
    if (a.out_idx != nullptr) {
        int32_t* out = a.out_idx + t * a.out_ts + h * a.out_hs;
        for (int s = lane; s < K; s += 32)
            out[s] = s < n ? selected_id(s, lo, hi, kp, all, buf_ids) : -1;
    }
    if (a.table) {
        const int width = K * kPagesPerBlock;
        int32_t* bt = a.sparse_bt + row * (int64_t)width;
        const int32_t* table = a.block_table + req * a.max_blocks;
        for (int e = lane; e < width; e += 32) {
            const int j = e >> 3;
            const int pg = e & 7;
            int32_t val = 0;
            if (j < n) {
                const int32_t b = selected_id(j, lo, hi, kp, all, buf_ids);
                if (b < a.max_blocks &&
                    (int64_t)b * kPageSize + (int64_t)pg * kSubPage < causal_len) {
                    const int32_t phys = __ldg(table + b);
                    report_status(a.status, pg == 0 && bad_phys_block(phys), BSA_STATUS_BAD_BLOCK_ID);
                    val = phys * kPagesPerBlock + pg;
                }
            }
            bt[e] = val;
        }
        int ctx = 0;
        for (int j = lane; j < n; j += 32) {
            const int32_t b = selected_id(j, lo, hi, kp, all, buf_ids);
            if (b < a.max_blocks) {
                const int64_t rem = causal_len - (int64_t)b * kPageSize;
                ctx += (int)(rem < kPageSize ? rem : kPageSize);
            }
        }
        ctx = __reduce_add_sync(kFull, ctx);
        if (lane == 0) a.sparse_ctx[row] = ctx;
    }
}

// Row geometry shared by both paths: causal bound, forced ranges, how many
// non-forced ids to select.
// rows < 2^31 (checked on the host), so t, h and req fit 32 bits; the causal
// length is at most seq_lens[req] <= INT32_MAX.
struct RowInfo {
    int32_t t, h, req, causal_len;
    int v, lo, hi, n, kp;
    bool all, need;
};

// Fused mode of a kernel instantiation: read from the arguments at run time,
// or fixed at compile time (plain select / fused select + table).
constexpr int kFusedRuntime = 0, kFusedNo = 1, kFusedYes = 2;

template <int FM>
__device__ __forceinline__ bool is_fused(const SelectArgs& a) {
    if constexpr (FM == kFusedRuntime) return a.fused;
    else return FM == kFusedYes;
}

// The per-row metadata word: num_valid_pages[t] (select) or seq_lens[req]
// (fused).  Split from row_info so the group path can load it one item early.
// x / d for x < 2^31 with the host's multiplier (see div_magic).
__device__ __forceinline__ uint32_t div_u31(uint32_t x, uint32_t mul, uint32_t shift) {
    return (__umulhi(x, mul) + x) >> shift;
}

template <int FM = kFusedRuntime>
__device__ __forceinline__ int32_t row_meta(const SelectArgs& a, int64_t row) {
    // rows < 2^31 (checked on the host)
    const uint32_t t32 = div_u31((uint32_t)row, a.h_mul, a.h_shift);
    if (is_fused<FM>(a)) return __ldg(a.seq_lens + div_u31(t32, a.dql_mul, a.dql_shift));
    return __ldg(a.num_valid_pages + t32);
}

template <int FM = kFusedRuntime>
__device__ __forceinline__ RowInfo row_info_from(const SelectArgs& a, int64_t row, int32_t meta) {
    RowInfo r;
    const uint32_t t32 = div_u31((uint32_t)row, a.h_mul, a.h_shift);
    r.t = (int32_t)t32;
    r.h = (int32_t)((uint32_t)row - t32 * (uint32_t)a.H);
    int64_t pages;
    r.causal_len = 0;
    r.req = 0;
    if (is_fused<FM>(a)) {
        const uint32_t req32 = div_u31(t32, a.dql_mul, a.dql_shift);
        r.req = (int32_t)req32;
        const int32_t lq = (int32_t)(t32 - req32 * (uint32_t)a.dql);
        const int64_t pos = (int64_t)meta - a.dql + lq;
        r.causal_len = (int32_t)(pos + 1 > 0 ? pos + 1 : 0);
        pages = ((int64_t)r.causal_len + kPageSize - 1) >> kLogPageSize;
    } else {
        pages = meta;
    }
    r.v = (int)(pages < 0 ? 0 : (pages > a.M ? a.M : pages));
    r.lo = a.num_init < r.v ? a.num_init : r.v;
    r.hi = max(r.v - a.num_local, r.lo);
    r.n = a.K < r.v ? a.K : r.v;
    r.kp = r.n - r.lo - (r.v - r.hi);         // non-forced ids to select
    r.all = r.kp >= r.hi - r.lo;              // every non-forced id fits
    r.need = r.kp > 0 && !r.all;
    return r;
}

__device__ __forceinline__ RowInfo row_info(const SelectArgs& a, int64_t row) {
    return row_info_from(a, row, row_meta(a, row));
}

// Ask L2 to fetch [addr, addr + bytes) (16-byte aligned, multiple of 16)
// ahead of use; no completion to wait for.
__device__ __forceinline__ void prefetch_l2(uintptr_t addr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(addr), "r"(bytes) : "memory");
}

// One work item (row, chunk) processed by a whole warp: the warp path, and
// the fallback of the group path for rows whose candidates overflow.  COH:
// the scores were written earlier in the same kernel, so they are read
// through L2 only.
template <bool BF16, int NV, int R, bool COH = false>
__device__ void warp_item(const KernelParams& P, int64_t row, int chunk, uint32_t* s_keys,
                          int32_t* s_ids, int lane) {
    using E = Elem<BF16>;
    constexpr int VEC = E::kVec;
    constexpr int S = E::kBytes;
    const SelectArgs& a = P.a;
    const int cap = P.cap;
    {
        const RowInfo ri = row_info(a, row);
        const int64_t t = ri.t, h = ri.h, causal_len = ri.causal_len, req = ri.req;
        const int lo = ri.lo, hi = ri.hi, n = ri.n, kp = ri.kp;
        const bool all = ri.all, need = ri.need;

        if (!need) {
            if (chunk == 0)
                write_outputs(P, row, t, h, n, lo, hi, kp, all, s_ids, causal_len, req, lane);
            return;
        }

        // ---- vector grid over the non-forced range [lo, hi) ----
        const char* row_ptr = reinterpret_cast<const char*>(a.scores) +
                              (t * a.token_stride + h * a.head_stride) * S;
        const uintptr_t a_lo = reinterpret_cast<uintptr_t>(row_ptr) + (uintptr_t)lo * S;
        const uintptr_t a_hi = reinterpret_cast<uintptr_t>(row_ptr) + (uintptr_t)hi * S;
        const uintptr_t v0 = a_lo & ~(uintptr_t)15;
        const int nvec = (int)((a_hi - v0 + 15) >> 4);
        const int base_id = lo - (int)((a_lo - v0) / S);
        const int nchunks = (nvec + P.vecs_per_chunk - 1) / P.vecs_per_chunk;
        if (chunk >= nchunks) return;
        const int k_begin = chunk * P.vecs_per_chunk;
        const int k_end = min(nvec, k_begin + P.vecs_per_chunk);
        if (!COH && k_end - k_begin > 32 * NV) {
            // more than one pass: bring the warp's whole range towards L2 at
            // once, 4 KB per lane, so that later passes do not wait on DRAM
            uintptr_t plo = v0 + ((uintptr_t)k_begin << 4);
            uintptr_t phi = v0 + ((uintptr_t)k_end << 4);
            if (plo < P.buf_lo) plo = (P.buf_lo + 15) & ~(uintptr_t)15;
            if (phi > P.buf_hi) phi = P.buf_hi & ~(uintptr_t)15;
            const uintptr_t at = plo + ((uintptr_t)lane << 12);
            if (at < phi) prefetch_l2(at, (uint32_t)min((uintptr_t)4096, phi - at));
        }

        Buf b{s_keys, s_ids, 0, 0u, false};
        // the largest theta of the earlier passes (raw, -1 = none): each is a
        // lower bound of the row's kp-th largest key, so it filters later passes
        int32_t th_run = -1;

        for (int pass = k_begin; pass < k_end && !b.closed; pass += 32 * NV) {
            // ---- load NV vectors per lane (masked outside [lo, hi)) ----
            uint4 w[NV];
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const int k = pass + j * 32 + lane;
                const uintptr_t addr = v0 + ((uintptr_t)k << 4);
                w[j] = make_uint4(E::kMaskWord, E::kMaskWord, E::kMaskWord, E::kMaskWord);
                if (k < k_end) {
                    if (addr >= a_lo && addr + 16 <= a_hi) {
                        w[j] = COH ? ld_cg_v4(reinterpret_cast<const void*>(addr))
                                   : ld_stream_v4(reinterpret_cast<const void*>(addr));
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            const int id = base_id + k * VEC + e;
                            if (id >= lo && id < hi) {
                                const char* ep = row_ptr + (int64_t)id * S;
                                E::set(w[j], e, COH ? E::load_one_cg(ep) : E::load_one(ep));
                            }
                        }
                    }
                }
            }

            // ---- representatives and the chunk's lower bound theta ----
            int32_t rep[R];
#pragma unroll
            for (int r = 0; r < R; ++r) rep[r] = INT32_MIN;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                int32_t q0, q1;
                if constexpr (BF16) {
                    const uint32_t pm = E::slot_pack_max(w[j]);
                    q0 = E::pack_lo(pm);
                    q1 = E::pack_hi(pm);
                } else {
                    q0 = E::even_max(w[j]);
                    q1 = E::odd_max(w[j]);
                }
                if constexpr (R == 1) {
                    rep[0] = max(rep[0], max(q0, q1));
                } else if constexpr (R == 2) {
                    rep[0] = max(rep[0], q0);
                    rep[1] = max(rep[1], q1);
                } else {
                    rep[(2 * j) % R] = max(rep[(2 * j) % R], q0);
                    rep[(2 * j + 1) % R] = max(rep[(2 * j + 1) % R], q1);
                }
            }
            // this pass's theta helps only if kp representatives lie above the
            // bounds already known (the entry bound's raw value and th_run);
            // otherwise the bit search is skipped and those bounds filter
            const int32_t known =
                max(b.kb >= E::kKeyOfPlusZero ? E::raw_of_nonneg_key(b.kb) : -1, th_run);
            int c0 = 0;
#pragma unroll
            for (int r = 0; r < R; ++r) c0 += rep[r] > known ? 1 : 0;
            c0 = __reduce_add_sync(kFull, c0);
            bool have_theta = c0 >= kp;
            int32_t theta = 0;
            if (have_theta) {
                for (int bit = E::kThetaTop; bit >= E::kThetaLow; --bit) {
                    const int32_t tt = theta | (1 << bit);
                    int c = 0;
#pragma unroll
                    for (int r = 0; r < R; ++r) c += rep[r] >= tt ? 1 : 0;
                    c = __reduce_add_sync(kFull, c);
                    if (c >= kp) theta = tt;
                }
                // fp32 searches the top 16 bits only, so theta may fall below
                // th_run
                theta = max(theta, th_run);
                th_run = theta;
            } else if (th_run >= 0) {
                have_theta = true;
                theta = th_run;
            }

            // ---- filter + append, one 32-vector slot at a time ----
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (pass + j * 32 >= k_end || b.closed) break;
                const int k = pass + j * 32 + lane;
                const int first_id = base_id + k * VEC;
                while (true) {
                    // Raw-space filter when the bound is a non-negative float.
                    const bool kb_nonneg = b.kb >= E::kKeyOfPlusZero;
                    const bool fast = have_theta || kb_nonneg;
                    int32_t th = 0;
                    if (fast) {
                        th = have_theta ? theta : 0;
                        if (kb_nonneg) th = max(th, E::raw_of_nonneg_key(b.kb));
                    }
                    unsigned m = 0;
                    if (fast) {
                        bool any;
                        if constexpr (BF16) {
                            any = E::pack_any_ge(E::slot_pack_max(w[j]), th);
                        } else {
                            any = max(E::even_max(w[j]), E::odd_max(w[j])) >= th;
                        }
                        if (any) {
#pragma unroll
                            for (int e = 0; e < VEC; ++e)
                                if (E::raw(w[j], e) >= th) m |= 1u << e;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            const int id = first_id + e;
                            if (id >= lo && id < hi && E::key(E::raw(w[j], e)) >= b.kb)
                                m |= 1u << e;
                        }
                    }
                    int pos;
                    if (!buf_try_append<E::kKeyBits, E::kKeyMax>(b, m, cap, kp, lane, pos)) {
                        if (b.closed) break;
                        continue;  // bound rose: recompute this slot's mask
                    }
                    if (pos >= 0) {
                        while (m) {
                            const int e = __ffs(m) - 1;
                            m &= m - 1;
                            b.keys[pos] = E::key(E::raw(w[j], e));
                            b.ids[pos] = first_id + e;
                            ++pos;
                        }
                    }
                    __syncwarp();
                    break;
                }
            }
        }
        if (b.n > kp) buf_compact<E::kKeyBits, E::kKeyMax>(b, kp, lane);

        if (nchunks > 1) {
            // ---- split row: publish this chunk, the last arriver merges ----
            const int64_t slot = row * P.chunks_per_row + chunk;
            uint32_t* wk = P.ws.keys + slot * a.K;
            int32_t* wi = P.ws.ids + slot * a.K;
            for (int e = lane; e < b.n; e += 32) {
                wk[e] = b.keys[e];
                wi[e] = b.ids[e];
            }
            if (lane == 0) P.ws.counts[slot] = b.n;
            __threadfence();
            __syncwarp();
            int ticket = 0;
            if (lane == 0) ticket = atomicAdd(P.ws.tickets + row, 1);
            ticket = __shfl_sync(kFull, ticket, 0);
            if (ticket != nchunks - 1) return;
            __threadfence();
            if (lane == 0) P.ws.tickets[row] = 0;  // ready for the next launch / replay
            b.n = 0;
            b.kb = 0;
            b.closed = false;
            for (int c = 0; c < nchunks && !b.closed; ++c) {
                const int64_t cs = row * P.chunks_per_row + c;
                const int cnt = __ldcg(P.ws.counts + cs);
                for (int g = 0; g < cnt && !b.closed; g += 32) {
                    const int e = g + lane;
                    const bool in = e < cnt;
                    const uint32_t key = in ? __ldcg(P.ws.keys + cs * a.K + e) : 0u;
                    const int32_t id = in ? __ldcg(P.ws.ids + cs * a.K + e) : 0;
                    while (true) {
                        const unsigned m = (in && key >= b.kb) ? 1u : 0u;
                        int pos;
                        if (!buf_try_append<E::kKeyBits, E::kKeyMax>(b, m, cap, kp, lane, pos)) {
                            if (b.closed) break;
                            continue;
                        }
                        if (pos >= 0 && m) {
                            b.keys[pos] = key;
                            b.ids[pos] = id;
                        }
                        __syncwarp();
                        break;
                    }
                }
            }
            if (b.n > kp) buf_compact<E::kKeyBits, E::kKeyMax>(b, kp, lane);
        }
        __syncwarp();
        write_outputs(P, row, t, h, n, lo, hi, kp, false, b.ids, causal_len, req, lane);
        __syncwarp();
    }
}

template <bool BF16, int NV, int R>
__global__ void __launch_bounds__(kThreads, 4) select_kernel(const KernelParams P) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint32_t* s_keys = reinterpret_cast<uint32_t*>(smem_raw) + (size_t)warp * P.cap * 2;
    int32_t* s_ids = reinterpret_cast<int32_t*>(s_keys + P.cap);
    const int64_t items = P.rows * P.chunks_per_row;
    const int64_t warps_total = (int64_t)gridDim.x * kWarpsPerCta;
    for (int64_t item = (int64_t)blockIdx.x * kWarpsPerCta + warp; item < items;
         item += warps_total) {
        int64_t row = item;
        int chunk = 0;
        if (P.chunks_per_row > 1) {
            row = (uint32_t)item / (uint32_t)P.chunks_per_row;
            chunk = (int)(item - row * P.chunks_per_row);
        }
        warp_item<BF16, NV, R>(P, row, chunk, s_keys, s_ids, lane);
    }
}


// ===========================================================================
// Group path: 4 lanes per row, 8 rows per warp.
//
// The warp path spends a full warp instruction on every per-row step (the
// threshold search, scans, the exact select), which bounds it by instruction
// issue long before HBM.  Here the 8 rows of a warp run those steps side by
// side, 4 lanes each:
//  1. pass 1: the 4 lanes of a row stream its non-forced range (64 contiguous
//     bytes per row per load instruction), store every 16-byte vector's
//     maximum (raw signed; fp32 keeps its top 16 bits) in shared memory, and
//     keep R representatives per lane;
//  2. theta = the K'-th largest of the row's 4R representatives (a 12-bit
//     search with 4-lane shuffle counts; coarse bits only make theta lower);
//  3. the vectors whose maximum reaches theta are queued warp-wide, so the
//     32 lanes share the detailed work of all 8 rows evenly;
//  4. the queued vectors are reloaded (L1/L2) and their elements >= theta are
//     appended to the row's candidate list as unique composite keys
//     (key << 16 | 0xFFFF - id for bf16, key << 32 | ~id for fp32), so their
//     order in the list does not matter;
//  5. each candidate's rank among the row's candidates decides selection;
//     the K' selected ids are sorted ascending by rank counting;
//  6. the 4 lanes write ids, and in fused mode the table and ctx.
// A row without a theta (fewer than K' non-negative representatives) takes
// every valid element as a candidate when they fit; a row whose candidates
// overflow the list is redone by the whole warp with the warp path.
// ===========================================================================

// Load vector k of a row's non-forced range.  Vectors that stick out of
// [lo, hi) (the first and the last) are loaded whole when they lie inside the
// score buffer, element by element otherwise, and the ids outside [lo, hi)
// are replaced by the mask pattern.
template <bool BF16>
__device__ __forceinline__ uint4 group_load_edge(const KernelParams& P, int k, uintptr_t v0,
                                                 int base_id, int lo, int hi,
                                                 const char* row_ptr) {
    using E = Elem<BF16>;
    constexpr int VEC = E::kVec;
    constexpr int S = E::kBytes;
    const uintptr_t addr = v0 + ((uintptr_t)k << 4);
    uint4 w;
    if (addr >= P.buf_lo && addr + 16 <= P.buf_hi) {
        w = __ldg(reinterpret_cast<const uint4*>(addr));
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int id = base_id + k * VEC + e;
            if (id < lo || id >= hi) E::set(w, e, (int32_t)E::kMaskWord);
        }
    } else {
        w = make_uint4(E::kMaskWord, E::kMaskWord, E::kMaskWord, E::kMaskWord);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int id = base_id + k * VEC + e;
            if (id >= lo && id < hi) E::set(w, e, E::load_one(row_ptr + (int64_t)id * S));
        }
    }
    return w;
}

// Two partial maxima of a vector (bf16: the two halves of the packed max;
// fp32: even and odd elements), raw signed.
template <bool BF16>
__device__ __forceinline__ void vec_max_pair(const uint4& w, int32_t& x0, int32_t& x1) {
    using E = Elem<BF16>;
    if constexpr (BF16) {
        const uint32_t pm = E::slot_pack_max(w);
        x0 = E::pack_lo(pm);
        x1 = E::pack_hi(pm);
    } else {
        x0 = E::even_max(w);
        x1 = E::odd_max(w);
    }
}

template <typename CK>
__device__ __forceinline__ CK make_ck(uint32_t key, int id);
template <>
__device__ __forceinline__ uint32_t make_ck<uint32_t>(uint32_t key, int id) {
    return (key << 16) | (0xFFFFu - (uint32_t)id);
}
template <>
__device__ __forceinline__ unsigned long long make_ck<unsigned long long>(uint32_t key, int id) {
    return ((unsigned long long)key << 32) | (0xFFFFFFFFu - (uint32_t)id);
}
// The low field of a composite: 0xFFFF - id (bf16) or 0xFFFFFFFF - id (fp32);
// larger means a lower id.
__device__ __forceinline__ uint32_t ck_low(uint32_t ck) { return ck & 0xFFFFu; }
__device__ __forceinline__ uint32_t ck_low(unsigned long long ck) { return (uint32_t)ck; }

template <typename T>
__device__ __forceinline__ T shfl_xor_any(T v, int m) {
    if constexpr (sizeof(T) == 8) {
        const uint32_t lo = __shfl_xor_sync(kFull, (uint32_t)v, m);
        const uint32_t hi = __shfl_xor_sync(kFull, (uint32_t)(v >> 32), m);
        return ((T)hi << 32) | lo;
    } else {
        return __shfl_xor_sync(kFull, v, m);
    }
}

// Bitonic sort, descending, of the 32 values a group of 4 lanes holds: lane
// q keeps positions 8q .. 8q + 7 in x[0..7].  Compare-exchanges within a lane
// stay in registers; those 8 or 16 positions apart use one shuffle per
// register.  Every lane of the warp must call this.
template <typename T>
__device__ __forceinline__ void group_sort32_desc(T (&x)[8], int q) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= 8) {
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const T y = shfl_xor_any(x[r], j >> 3);
                    const int p = q * 8 + r;
                    const bool keep_max = ((p & j) == 0) == ((p & k) == 0);
                    const T mx = x[r] > y ? x[r] : y;
                    const T mn = x[r] > y ? y : x[r];
                    x[r] = keep_max ? mx : mn;
                }
            } else {
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    if ((r & j) == 0) {
                        const int p = q * 8 + r;
                        const bool desc = (p & k) == 0;
                        const T a = x[r], b = x[r | j];
                        const T mx = a > b ? a : b;
                        const T mn = a > b ? b : a;
                        x[r] = desc ? mx : mn;
                        x[r | j] = desc ? mn : mx;
                    }
                }
            }
        }
    }
}

// Bitonic sort, descending, of the 16 values a group of 4 lanes holds: lane
// q keeps positions 4q .. 4q + 3 in x[0..3].
template <typename T>
__device__ __forceinline__ void group_sort16_desc(T (&x)[4], int q) {
#pragma unroll
    for (int k = 2; k <= 16; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j >= 4) {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const T y = shfl_xor_any(x[r], j >> 2);
                    const int p = q * 4 + r;
                    const bool keep_max = ((p & j) == 0) == ((p & k) == 0);
                    const T mx = x[r] > y ? x[r] : y;
                    const T mn = x[r] > y ? y : x[r];
                    x[r] = keep_max ? mx : mn;
                }
            } else {
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    if ((r & j) == 0) {
                        const int p = q * 4 + r;
                        const bool desc = (p & k) == 0;
                        const T a = x[r], b = x[r | j];
                        const T mx = a > b ? a : b;
                        const T mn = a > b ? b : a;
                        x[r] = desc ? mx : mn;
                        x[r | j] = desc ? mn : mx;
                    }
                }
            }
        }
    }
}

// x[idx] for a register array and a runtime index (a chain of selects).
template <typename T, int N>
__device__ __forceinline__ T pick(const T (&x)[N], int idx) {
    T v = x[0];
#pragma unroll
    for (int r = 1; r < N; ++r) v = idx == r ? x[r] : v;
    return v;
}

__device__ __forceinline__ int32_t group_sel(int j, const RowInfo& r, bool all,
                                             const int32_t* sorted) {
    if (all || j < r.lo) return j;
    if (j - r.lo < r.kp) return sorted[j - r.lo];
    return r.hi + (j - r.lo - r.kp);
}

// Outputs of one row by its LANES lanes: lane q owns the output slots (=
// blocks) q, q + LANES, q + 2 LANES, ..., so that at each step the row's lanes
// write adjacent 32-byte table slots; it writes their ids, their 8 table
// entries each (one 32-byte store) and their part of ctx.  Every lane of the warp calls
// this (ctx is summed with shuffles inside each row's lanes); `write` masks
// the stores.
template <int LANES, int FM = kFusedRuntime>
__device__ void group_write_outputs(const KernelParams& P, int64_t row, const RowInfo& r,
                                    bool all, const int32_t* sorted, int q, bool write) {
    const SelectArgs& a = P.a;
    const int K = a.K;
    const bool fused = is_fused<FM>(a);
    int ctx = 0;
    if (write) {
        int32_t* out = a.out_idx != nullptr
                           ? a.out_idx + (int64_t)r.t * a.out_ts + (int64_t)r.h * a.out_hs
                           : nullptr;
        const int width = K * kPagesPerBlock;
        int32_t* bt = fused ? a.sparse_bt + row * (int64_t)width : nullptr;
        const int32_t* table = fused ? a.block_table + (int64_t)r.req * a.max_blocks : nullptr;
        const bool vec_ok = ((reinterpret_cast<uintptr_t>(bt)) & 31) == 0;  // 32-byte slots
        // 8 slots at a time: ids first, then all table gathers in flight
        // together, then the stores
        const int per = (K + LANES - 1) / LANES;
        for (int u0 = 0; u0 < per; u0 += 8) {
            int32_t bs[8], phys[8];
            bool okb[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = q + LANES * (u0 + u);
                bs[u] = (j < K && j < r.n) ? group_sel(j, r, all, sorted) : -1;
                okb[u] = bt != nullptr && bs[u] >= 0 && bs[u] < a.max_blocks;
                phys[u] = 0;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (okb[u]) phys[u] = __ldg(table + bs[u]);
            if (a.status != nullptr) {
                bool bad = false;
#pragma unroll
                for (int u = 0; u < 8; ++u) bad |= okb[u] && bad_phys_block(phys[u]);
                report_status(a.status, bad, BSA_STATUS_BAD_BLOCK_ID);
            }
            if (out != nullptr) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = q + LANES * (u0 + u);
                    if (j < K) out[j] = bs[u];
                }
            }
            if (bt == nullptr) continue;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = q + LANES * (u0 + u);
                if (j >= K) break;
                int v[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if (okb[u]) {
                    const int rem = (int)min(r.causal_len - (int64_t)bs[u] * kPageSize,
                                             (int64_t)kPageSize);
                    const int32_t phys8 = phys[u] * kPagesPerBlock;
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = e * kSubPage < rem ? phys8 + e : 0;
                    ctx += rem;
                }
                int32_t* dst = bt + 8 * j;
                if (vec_ok) {
                    st_v8(dst, v);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) dst[e] = v[e];
                }
            }
        }
    }
    if (!fused) return;
#pragma unroll
    for (int m = 1; m < LANES; m <<= 1) ctx += __shfl_xor_sync(kFull, ctx, m);
    if (write && q == 0) a.sparse_ctx[row] = ctx;
}

template <bool BF16, int R, bool SMALLK>
__global__ void __launch_bounds__(kThreads, 3) group_select_kernel(const KernelParams P) {
    using E = Elem<BF16>;
    using CK = typename std::conditional<BF16, uint32_t, unsigned long long>::type;
    using G = GroupSmem<CK>;
    constexpr int VEC = E::kVec;
    constexpr int S = E::kBytes;
    constexpr int H2 = R / 2;  // representative pairs per lane (divides 4)
    static_assert(R == 2 || R == 4 || R == 8, "R must be 2, 4 or 8");
    static_assert(kGroupCand == 32, "the candidate sort holds 32 values");
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane >> 2;
    const int q = lane & 3;
    G& sm = *reinterpret_cast<G*>(smem_raw + (size_t)warp * sizeof(G));
    const SelectArgs& a = P.a;
    const int64_t ngroups = (P.rows + kGroupRows - 1) / kGroupRows;
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerCta;

    int64_t wg = (int64_t)blockIdx.x * kWarpsPerCta + warp;
    int32_t meta = 0;
    if (wg < ngroups && wg * kGroupRows + g < P.rows) meta = row_meta(a, wg * kGroupRows + g);
    for (; wg < ngroups; wg += stride) {
        const int64_t row = wg * kGroupRows + g;
        const bool active = row < P.rows;
        // metadata of the next item, loaded now and used after pass 1
        const int64_t nrow = (wg + stride) * kGroupRows + g;
        const bool nactive = wg + stride < ngroups && nrow < P.rows;
        const int32_t nmeta = nactive ? row_meta(a, nrow) : 0;
        RowInfo r{};
        r.all = true;
        if (active) r = row_info_from(a, row, meta);
        meta = nmeta;
        const bool need = active && r.need;

        // ---- geometry of the non-forced range [lo, hi) ----
        const char* row_ptr = nullptr;
        uintptr_t v0 = 0;
        int nvec = 0, base_id = 0;
        if (need) {
            row_ptr = reinterpret_cast<const char*>(a.scores) +
                      (r.t * a.token_stride + r.h * a.head_stride) * S;
            const uintptr_t a_lo = reinterpret_cast<uintptr_t>(row_ptr) + (uintptr_t)r.lo * S;
            const uintptr_t a_hi = reinterpret_cast<uintptr_t>(row_ptr) + (uintptr_t)r.hi * S;
            v0 = a_lo & ~(uintptr_t)15;
            nvec = (int)((a_hi - v0 + 15) >> 4);
            base_id = r.lo - (int)((a_lo - v0) / S);
        }

        // ---- pass 1: vector maxima and representatives ----
        // Step 0 holds vectors 0..3 (the first one is an edge), the interior
        // vectors 4 .. nvec-2 need no masking, the last one is an edge.
        int32_t rep[R];
#pragma unroll
        for (int x = 0; x < R; ++x) rep[x] = INT32_MIN;
        auto take = [&](const uint4& w, int k, int slot) {
            int32_t x0, x1;
            vec_max_pair<BF16>(w, x0, x1);
            const int32_t m = max(x0, x1);
            sm.vmax[g][q][(k - q) >> 2] = (int16_t)(BF16 ? m : (m >> 16));
            rep[(slot % H2) * 2] = max(rep[(slot % H2) * 2], x0);
            rep[(slot % H2) * 2 + 1] = max(rep[(slot % H2) * 2 + 1], x1);
        };
        if (need && q < nvec) {
            take(group_load_edge<BF16>(P, q, v0, base_id, r.lo, r.hi, row_ptr), q, 0);
        }
        // interior vectors k = q + 4 i, i >= 1, k <= nvec - 2
        const int n_int = need ? max(0, (nvec - 2 - q) / kGroupLanes) : 0;
        for (int i0 = 1; i0 <= n_int; i0 += 4) {
            uint4 w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u;
                const uintptr_t addr = v0 + ((uintptr_t)(q + kGroupLanes * i) << 4);
                if (i <= n_int) w[u] = __ldg(reinterpret_cast<const uint4*>(addr));
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u;
                if (i <= n_int) take(w[u], q + kGroupLanes * i, u + 1);
            }
        }
        if (need && nvec > kGroupLanes && (nvec - 1) % kGroupLanes == q) {
            take(group_load_edge<BF16>(P, nvec - 1, v0, base_id, r.lo, r.hi, row_ptr), nvec - 1,
                 3);
        }
        // the rows of this warp's next item start streaming into L2 while
        // this item is being selected
        if (q == 0 && nactive) {
            const RowInfo nr = row_info_from(a, nrow, nmeta);
            if (nr.need) {
                const uintptr_t nrp = reinterpret_cast<uintptr_t>(a.scores) +
                                      (uintptr_t)((nr.t * a.token_stride + nr.h * a.head_stride) * S);
                const uintptr_t nlo = (nrp + (uintptr_t)nr.lo * S) & ~(uintptr_t)15;
                uintptr_t nhi = (nrp + (uintptr_t)nr.hi * S + 15) & ~(uintptr_t)15;
                if (nhi > P.buf_hi) nhi = P.buf_hi & ~(uintptr_t)15;
                if (nlo >= P.buf_lo && nhi > nlo) prefetch_l2(nlo, (uint32_t)(nhi - nlo));
            }
        }

        // ---- theta: the K'-th largest representative of the row ----
        // 12-bit search from the top (bf16: 1/16-binade resolution; fp32 uses
        // its top 12 bits); the bits left at zero only lower theta
        constexpr int kTop = BF16 ? 14 : 30;
        constexpr int kLow = BF16 ? 3 : 19;
        int c0 = 0;
#pragma unroll
        for (int x = 0; x < R; ++x) c0 += rep[x] >= 0 ? 1 : 0;
        c0 += __shfl_xor_sync(kFull, c0, 1);
        c0 += __shfl_xor_sync(kFull, c0, 2);
        const bool fast = need && c0 >= r.kp;
        int32_t theta = 0;
        for (int bit = kTop; bit >= kLow; --bit) {
            const int32_t tt = theta | (1 << bit);
            int c = 0;
#pragma unroll
            for (int x = 0; x < R; ++x) c += rep[x] >= tt ? 1 : 0;
            c += __shfl_xor_sync(kFull, c, 1);
            c += __shfl_xor_sync(kFull, c, 2);
            if (c >= r.kp) theta = tt;
        }
        const bool ovf0 = need && !fast && (r.hi - r.lo) > kGroupCand;
        if (q == 0) {
            sm.ccount[g] = 0;
            sm.ovf[g] = ovf0 ? 1 : 0;
            GroupRowDesc d;
            d.v0 = v0;
            d.row_ptr = reinterpret_cast<uintptr_t>(row_ptr);
            d.base_id = base_id;
            d.lo = r.lo;
            d.hi = r.hi;
            d.theta = theta;
            d.fast = fast ? 1 : 0;
            d.nvec = nvec;
            sm.desc[g] = d;
        }
        const int32_t th16 = BF16 ? theta : (theta >> 16);

        // ---- queue the vectors that can hold candidates ----
        // Each lane marks its hot vectors in a bitmask (8 maxima per 16-byte
        // shared load), the warp scans the counts, and every lane writes its
        // entries contiguously: the queue's order does not matter.
        const int my_steps = (need && !ovf0) ? (nvec - q + kGroupLanes - 1) / kGroupLanes : 0;
        unsigned long long hot = 0;
        for (int i0 = 0; i0 < my_steps; i0 += 8) {
            const uint4 pk = *reinterpret_cast<const uint4*>(&sm.vmax[g][q][i0]);
            const uint32_t wv[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int32_t vm = (int32_t)(int16_t)(uint16_t)(wv[u >> 1] >> ((u & 1) * 16));
                if (i0 + u < my_steps && (!fast || vm >= th16)) hot |= 1ull << (i0 + u);
            }
        }
        int qtotal;
        int qpos = warp_excl_scan(__popcll(hot), lane, qtotal);
        while (hot) {
            const int i = __ffsll((long long)hot) - 1;
            hot &= hot - 1;
            sm.q.queue[qpos++] = (uint16_t)((g << 13) | (q + kGroupLanes * i));
        }
        const int qn = qtotal;
        __syncwarp();

        // ---- candidates from the queued vectors, 32 at a time ----
        for (int base = 0; base < qn; base += 32) {
            const int e = base + lane;
            if (e < qn) {
                const int ent = sm.q.queue[e];
                const int gg = ent >> 13;
                const int k = ent & 0x1FFF;
                const GroupRowDesc d = sm.desc[gg];
                uint4 w;
                if (k == 0 || k == d.nvec - 1)
                    w = group_load_edge<BF16>(P, k, (uintptr_t)d.v0, d.base_id, d.lo, d.hi,
                                              reinterpret_cast<const char*>(d.row_ptr));
                else
                    w = __ldg(reinterpret_cast<const uint4*>((uintptr_t)d.v0 + ((uintptr_t)k << 4)));
                const int first_id = d.base_id + k * VEC;
                unsigned m = 0;
                if (d.fast) {
#pragma unroll
                    for (int x = 0; x < VEC; ++x)
                        if (E::raw(w, x) >= d.theta) m |= 1u << x;
                } else {
#pragma unroll
                    for (int x = 0; x < VEC; ++x) {
                        const int id = first_id + x;
                        if (id >= d.lo && id < d.hi) m |= 1u << x;
                    }
                }
                const int nc = __popc(m);
                if (nc) {
                    int p = atomicAdd(&sm.ccount[gg], nc);
                    if (p + nc <= kGroupCand) {
                        while (m) {
                            const int x = __ffs(m) - 1;
                            m &= m - 1;
                            sm.cand[gg][p++] = make_ck<CK>(E::key(E::raw(w, x)), first_id + x);
                        }
                    } else {
                        sm.ovf[gg] = 1;
                    }
                }
            }
        }
        __syncwarp();

        // ---- exact select: sort the row's candidates, keep the first K' ----
        const bool ovf = sm.ovf[g] != 0;
        const int cn = min(sm.ccount[g], kGroupCand);
        const bool sel_ok = need && !ovf;
        CK x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int pos = q * 8 + u;
            x[u] = (sel_ok && pos < cn) ? sm.cand[g][pos] : (CK)0;
        }
        group_sort32_desc<CK>(x, q);
        // keep positions < K'; re-sort the kept ids ascending (descending low field)
        constexpr uint32_t kLowMax = BF16 ? 0xFFFFu : 0xFFFFFFFFu;
        if (SMALLK) {
            // K' <= 16: positions 0..15 live in lanes 0 and 1; lane q takes 4q .. 4q+3
            uint32_t y[4];
            const int src = (g << 2) | (q >> 1);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                // position 4q + u is register 4 (q & 1) + u of lane q >> 1
                const uint32_t got0 = __shfl_sync(kFull, ck_low(x[u]), src);
                const uint32_t got1 = __shfl_sync(kFull, ck_low(x[u + 4]), src);
                y[u] = (q * 4 + u < r.kp) ? ((q & 1) ? got1 : got0) : 0u;
            }
            group_sort16_desc<uint32_t>(y, q);
            __syncwarp();
            if (sel_ok) {
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int pos = q * 4 + u;
                    if (pos < r.kp) sm.q.s.sorted[g][pos] = (int32_t)(kLowMax - y[u]);
                }
            }
        } else {
            uint32_t y[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) y[u] = (q * 8 + u < r.kp) ? ck_low(x[u]) : 0u;
            group_sort32_desc<uint32_t>(y, q);
            __syncwarp();
            if (sel_ok) {
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int pos = q * 8 + u;
                    if (pos < r.kp) sm.q.s.sorted[g][pos] = (int32_t)(kLowMax - y[u]);
                }
            }
        }
        __syncwarp();

        // ---- outputs ----
        group_write_outputs<kGroupLanes>(P, row, r, r.all, sm.q.s.sorted[g], q,
                                         active && (!need || !ovf));

        // ---- rows whose candidates overflowed: the whole warp redoes them ----
        unsigned fb = __ballot_sync(kFull, q == 0 && need && ovf);
        __syncwarp();
        while (fb) {
            const int bit = __ffs(fb) - 1;
            fb &= fb - 1;
            const int64_t frow = wg * kGroupRows + (bit >> 2);
            uint32_t* s_keys = reinterpret_cast<uint32_t*>(&sm);
            warp_item<BF16, 4, 2>(P, frow, 0, s_keys, reinterpret_cast<int32_t*>(s_keys + P.cap),
                                  lane);
            __syncwarp();
        }
        __syncwarp();
    }
}


// ===========================================================================
// Pair path: 2 lanes per row, 16 rows per warp.
//
// Same algorithm as the group path with half the lanes per row, so that the
// fixed per-row steps (threshold search, sorts, outputs) cover 16 rows per
// warp instruction, and with 32-byte chunks (one 256-bit load per lane, a
// row's pair reads 64 contiguous bytes per instruction).
//
// Elements become signed order-preserving keys as they are loaded: a
// negative value has its low 15 (bf16) or 31 (fp32) bits flipped, after which
// signed integer order is totalOrder.  Maxima, representatives and the
// threshold therefore work for rows of any sign.  Representatives stay
// packed: bf16 keeps 16 per lane in 8 registers updated with max.s16x2.
//
// A row whose candidates overflow the 32-entry list is redone by the whole
// warp on the warp path (no candidate limit) before the warp moves on.
// ===========================================================================

__device__ __forceinline__ void ld32(uintptr_t addr, uint32_t (&w)[8]) {
    asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
          "=r"(w[7])
        : "l"(addr));
}

// Signed order-preserving key of one raw element (sign-extended to int32).
template <bool BF16>
__device__ __forceinline__ int32_t key_of_raw(int32_t raw) {
    if constexpr (BF16) return raw ^ ((raw >> 15) & 0x7FFF);
    else return raw ^ ((raw >> 31) & 0x7FFFFFFF);
}

// 0xFFFF in each 16-bit half of x whose sign bit is set (prmt with the
// sign-replicate selector).
__device__ __forceinline__ uint32_t sign_mask16(uint32_t x) {
    uint32_t m;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(m) : "r"(x), "r"(0u), "n"(0xBB99));
    return m;
}

// The same on a whole 32-byte chunk, in place (bf16: two keys per word).
template <bool BF16>
__device__ __forceinline__ void chunk_to_keys(uint32_t (&w)[8]) {
#pragma unroll
    for (int x = 0; x < 8; ++x) {
        if constexpr (BF16) {
            w[x] ^= sign_mask16(w[x]) & 0x7FFF7FFFu;
        } else {
            w[x] ^= (uint32_t)((int32_t)w[x] >> 31) & 0x7FFFFFFFu;
        }
    }
}

template <bool BF16>
__device__ __forceinline__ int32_t chunk_raw(const uint32_t (&w)[8], int e) {
    if constexpr (BF16) return (int32_t)(int16_t)(uint16_t)(w[e >> 1] >> ((e & 1) * 16));
    else return (int32_t)w[e];
}

template <bool BF16>
__device__ __forceinline__ void chunk_set(uint32_t (&w)[8], int e, int32_t raw) {
    if constexpr (BF16) {
        const int sh = (e & 1) * 16;
        w[e >> 1] = (w[e >> 1] & ~(0xFFFFu << sh)) | (((uint32_t)raw & 0xFFFFu) << sh);
    } else {
        w[e] = (uint32_t)raw;
    }
}

// Chunk k of a row's non-forced range as keys, with ids outside [lo, hi) set
// to the smallest key (0x8000 / 0x80000000).
template <bool BF16>
__device__ __forceinline__ void pair_load_edge(const KernelParams& P, int k, uintptr_t c0,
                                               int base_id, int lo, int hi,
                                               const char* row_ptr, uint32_t (&w)[8]) {
    using E = Elem<BF16>;
    constexpr int S = E::kBytes;
    constexpr int CE = 32 / S;
    const uintptr_t addr = c0 + ((uintptr_t)k << 5);
    if (addr >= P.buf_lo && addr + 32 <= P.buf_hi) {
        ld32(addr, w);
        chunk_to_keys<BF16>(w);
        const int d0 = base_id + k * CE - lo;   // first id of the chunk, relative to lo
        const uint32_t span = (uint32_t)(hi - lo);
        if (d0 < 0 || (uint32_t)(d0 + CE) > span) {
            // element e is kept iff 0 <= d0 + e < hi - lo; one mask word per word
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                if constexpr (BF16) {
                    const uint32_t keep = ((uint32_t)(d0 + 2 * x) < span ? 0x0000FFFFu : 0u) |
                                          ((uint32_t)(d0 + 2 * x + 1) < span ? 0xFFFF0000u : 0u);
                    w[x] = (w[x] & keep) | (E::kMaskWord & ~keep);
                } else {
                    if ((uint32_t)(d0 + x) >= span) w[x] = E::kMaskWord;
                }
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = E::kMaskWord;
#pragma unroll
        for (int e = 0; e < CE; ++e) {
            const int id = base_id + k * CE + e;
            if (id >= lo && id < hi)
                chunk_set<BF16>(w, e, key_of_raw<BF16>(E::load_one(row_ptr + (int64_t)id * S)));
        }
    }
}

// One bit per int16 half of NW packed words: bit e set when half e >= t
// (signed), for t > -32768.  max.s16x2(x, t - 1) differs from t - 1 iff x >= t.
template <int NW>
__device__ __forceinline__ uint32_t ge_bits16(const uint32_t (&w)[NW], int32_t t) {
    const uint32_t t2 = ((uint32_t)(t - 1) & 0xFFFFu) * 0x10001u;
    uint32_t b[NW];
#pragma unroll
    for (int x = 0; x < NW; ++x) b[x] = min_u16x2(max_s16x2(w[x], t2) ^ t2, 0x00010001u);
    uint32_t bits = 0;
#pragma unroll
    for (int x = 0; x < NW; x += 2) {
        // bytes: halves 2x, 2x+1, 2x+2, 2x+3 as 0/1, folded into 4 bits
        const uint32_t v4 = __byte_perm(b[x], b[x + 1], 0x6420);
        bits |= ((v4 * 0x01020408u) >> 24) << (2 * x);
    }
    return bits;
}

// ge_bits16<8> with the bits in another order: bit x (x < 8) is element 2x
// and bit 8 + x is element 2x + 1 of the chunk; shifts and adds replace the
// byte gathers.
__device__ __forceinline__ uint32_t ge_bits16_perm(const uint32_t (&w)[8], int32_t t) {
    const uint32_t t2 = ((uint32_t)(t - 1) & 0xFFFFu) * 0x10001u;
    uint32_t c = 0;
#pragma unroll
    for (int x = 0; x < 8; ++x) c += min_u16x2(max_s16x2(w[x], t2) ^ t2, 0x00010001u) << x;
    return (c & 0xFFu) | ((c >> 8) & 0xFF00u);
}

// Element of a bf16 chunk named by bit b of ge_bits16_perm.
__device__ __forceinline__ int perm_elem(int b) { return ((b & 7) << 1) | (b >> 3); }

// Sorting 16 sixteen-bit values packed two per word: value r sits in word
// r & 7, low half for r < 8 and high half for r >= 8.  One max/min of two
// words compares the two columns at once.  SG selects signed or unsigned
// order.
template <bool SG>
__device__ __forceinline__ uint32_t hmax(uint32_t a, uint32_t b) {
    return SG ? max_s16x2(a, b) : max_u16x2(a, b);
}
template <bool SG>
__device__ __forceinline__ uint32_t hmin(uint32_t a, uint32_t b) {
    return SG ? min_s16x2(a, b) : min_u16x2(a, b);
}

// Each 16-bit half of every word: low half <- max of the two, high <- min.
template <bool SG>
__device__ __forceinline__ uint32_t hsplit(uint32_t t) {
    const uint32_t sw = __byte_perm(t, 0, 0x1032);
    return __byte_perm(hmax<SG>(t, sw), hmin<SG>(t, sw), 0x7610);
}

// Descending half-cleaners j = 4, 2, 1 on both columns: each column, bitonic
// on entry, leaves sorted.
template <bool SG>
__device__ __forceinline__ void hclean8_desc(uint32_t (&w)[8]) {
#pragma unroll
    for (int j = 4; j > 0; j >>= 1) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            if ((r & j) == 0) {
                const uint32_t a = w[r], b = w[r | j];
                w[r] = hmax<SG>(a, b);
                w[r | j] = hmin<SG>(a, b);
            }
        }
    }
}

// The 16 packed values sorted descending (positions 0..7 in the low halves).
template <bool SG>
__device__ __forceinline__ void packed_sort16_desc(uint32_t (&w)[8]) {
    // each column (8 values) by a bitonic network on whole words
#pragma unroll
    for (int k = 2; k <= 8; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                if ((r & j) == 0) {
                    const bool desc = (r & k) == 0 || k == 8;
                    const uint32_t a = w[r], b = w[r | j];
                    const uint32_t mx = hmax<SG>(a, b), mn = hmin<SG>(a, b);
                    w[r] = desc ? mx : mn;
                    w[r | j] = desc ? mn : mx;
                }
            }
        }
    }
    // merge the sorted columns A (low) and B (high): max(A[i], B[7 - i]) are
    // the top 8 as a bitonic sequence, the minima the bottom 8
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = __byte_perm(w[i], w[7 - i], 0x7610);
        const uint32_t b = __byte_perm(w[7 - i], w[i], 0x7610);
        w[i] = hsplit<SG>(a);
        w[7 - i] = hsplit<SG>(b);
    }
    hclean8_desc<SG>(w);
}

// The 16 largest of the 32 packed values a lane pair holds, sorted
// descending, in both lanes' registers (the packed form of pair_top16_desc).
template <bool SG>
__device__ __forceinline__ void packed_pair_top16_desc(uint32_t (&w)[8]) {
    packed_sort16_desc<SG>(w);
    // c[r] = max(a[r], b[15 - r]): for word i, the partner's word 7 - i with
    // its halves swapped
    uint32_t y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __shfl_xor_sync(0xffffffffu, w[7 - i], 1);
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = hmax<SG>(w[i], __byte_perm(y[i], 0, 0x1032));
    // c is bitonic: half-cleaner j = 8 (low vs high half of each word), then
    // j = 4, 2, 1 within the columns
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = hsplit<SG>(w[i]);
    hclean8_desc<SG>(w);
}

// Bitonic sort, descending, of the 32 values a lane pair holds: lane s keeps
// positions 16 s .. 16 s + 15 in x[0..15].  Every lane of the warp calls it.
template <typename T>
__device__ __forceinline__ void pair_sort32_desc(T (&x)[16], int s) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            if (j == 16) {
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const T y = shfl_xor_any(x[r], 1);
                    const T mx = x[r] > y ? x[r] : y;
                    const T mn = x[r] > y ? y : x[r];
                    x[r] = s == 0 ? mx : mn;  // k == 32: descending, lane 0 is the upper half
                }
            } else {
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    if ((r & j) == 0) {
                        const bool desc = k < 16 ? ((r & k) == 0) : (k == 32 || s == 0);
                        const T a = x[r], b = x[r | j];
                        const T mx = a > b ? a : b;
                        const T mn = a > b ? b : a;
                        x[r] = desc ? mx : mn;
                        x[r | j] = desc ? mn : mx;
                    }
                }
            }
        }
    }
}

// Bitonic sort, descending, of 16 values in one lane's registers.
template <typename T>
__device__ __forceinline__ void lane_sort16_desc(T (&x)[16]) {
#pragma unroll
    for (int k = 2; k <= 16; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                if ((r & j) == 0) {
                    const bool desc = (r & k) == 0 || k == 16;
                    const T a = x[r], b = x[r | j];
                    const T mx = a > b ? a : b;
                    const T mn = a > b ? b : a;
                    x[r] = desc ? mx : mn;
                    x[r | j] = desc ? mn : mx;
                }
            }
        }
    }
}

// The 16 largest of the 32 values a lane pair holds, descending, in lane 0's
// x[0..15] (lane 1's registers end up unspecified).  Each lane sorts its 16;
// lane 0 then keeps max(a[r], b[15 - r]) of its list a and the partner's list
// b, a bitonic sequence holding the top 16, and merges it.
template <typename T>
__device__ __forceinline__ void pair_top16_desc(T (&x)[16]) {
    lane_sort16_desc<T>(x);
    T y[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) y[r] = shfl_xor_any(x[15 - r], 1);
#pragma unroll
    for (int r = 0; r < 16; ++r) x[r] = x[r] > y[r] ? x[r] : y[r];
#pragma unroll
    for (int j = 8; j > 0; j >>= 1) {
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            if ((r & j) == 0) {
                const T a = x[r], b = x[r | j];
                x[r] = a > b ? a : b;
                x[r | j] = a > b ? b : a;
            }
        }
    }
}

template <bool BF16, bool SMALLK, int FM>
// The plain bf16 select needs fewer registers than the fused kernel, whose
// table epilogue holds 8 gathers in flight: more of its CTAs fit on an SM.
__global__ void __launch_bounds__(kPairWarps * 32,
                                  FM == kFusedNo && BF16 ? kPairCtasSelect : kPairCtas)
    pair_select_kernel(const KernelParams P) {
    using E = Elem<BF16>;
    using CK = typename std::conditional<BF16, uint32_t, unsigned long long>::type;
    using G = PairSmem<CK>;
    constexpr int S = E::kBytes;
    constexpr int CE = 32 / S;                 // elements per 32-byte chunk
    constexpr uint32_t kFlip = BF16 ? 0x8000u : 0x80000000u;  // signed key -> unsigned key
    constexpr uint32_t kLowMax = BF16 ? 0xFFFFu : 0xFFFFFFFFu;
    constexpr int32_t kKeyMin = BF16 ? -32768 : INT32_MIN;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int p = lane >> 1;   // row of the warp's item
    const int s = lane & 1;    // lane within the row's pair
    G& sm = *reinterpret_cast<G*>(smem_raw + (size_t)warp * sizeof(G));
    const SelectArgs& a = P.a;
    // rows < 2^31 (checked on the host), so items and the policy's grid fit int
    const int nitems = (int)((P.rows + kPairRows - 1) / kPairRows);
    const int stride = (int)gridDim.x * kPairWarps;

    int it = (int)blockIdx.x * kPairWarps + warp;
    int32_t meta = 0;
    if (it < nitems && (int64_t)it * kPairRows + p < P.rows) meta = row_meta<FM>(a, (int64_t)it * kPairRows + p);
    for (; it < nitems; it += stride) {
        const int64_t row = (int64_t)it * kPairRows + p;
        const bool active = row < P.rows;
        const int64_t nrow = ((int64_t)it + stride) * kPairRows + p;
        const bool nactive = (int64_t)it + stride < nitems && nrow < P.rows;
        const int32_t nmeta = nactive ? row_meta<FM>(a, nrow) : 0;
        RowInfo r{};
        r.all = true;
        if (active) r = row_info_from<FM>(a, row, meta);
        const int32_t cur_meta = meta;
        meta = nmeta;
        // a row whose range exceeds 2 KB (a wider buffer) goes to the list of
        // the second, wide-path launch
        const bool longr = P.long_list != nullptr && active && r.need &&
                           (int64_t)(r.hi - r.lo) * S > kGroupMaxBytes;
        if (longr && s == 0) P.long_list[atomicAdd(P.long_count, 1u)] = (int32_t)row;
        const bool need = active && r.need && !longr;

        // ---- geometry of the non-forced range [lo, hi), 32-byte chunks ----
        const char* row_ptr = nullptr;
        uintptr_t c0 = 0;
        int nchunk = 0, base_id = 0;
        if (need) {
            row_ptr = reinterpret_cast<const char*>(a.scores) +
                      ((int64_t)r.t * a.token_stride + (int64_t)r.h * a.head_stride) * S;
            const uintptr_t a_lo = reinterpret_cast<uintptr_t>(row_ptr) + (uintptr_t)r.lo * S;
            const uintptr_t a_hi = reinterpret_cast<uintptr_t>(row_ptr) + (uintptr_t)r.hi * S;
            c0 = a_lo & ~(uintptr_t)31;
            nchunk = (int)((a_hi - c0 + 31) >> 5);
            base_id = r.lo - (int)((a_lo - c0) / S);
            // one bulk request brings the whole range towards L2 while the
            // lanes' own loads walk it in batches
            if (s == 0) {
                const uintptr_t plo = c0 < P.buf_lo ? (P.buf_lo + 15) & ~(uintptr_t)15 : c0;
                uintptr_t phi = c0 + ((uintptr_t)nchunk << 5);
                if (phi > P.buf_hi) phi = P.buf_hi & ~(uintptr_t)15;
                if (phi > plo) prefetch_l2(plo, (uint32_t)(phi - plo));
            }
        }

        // ---- pass 1: chunk maxima and representatives ----
        // Step i covers chunks 4i .. 4i+3 (one 128-byte line of the row): lane
        // s takes chunks 4i + 2s and 4i + 2s + 1.  The step's two chunk maxima
        // go to vmax2[i][lane] in one store; representatives: 4 classes (by
        // step and chunk parity) x 4 disjoint element subsets.
        uint32_t rp[8];   // bf16: packed pairs; fp32 uses rq
        int32_t rq[16];
#pragma unroll
        for (int x = 0; x < 8; ++x) rp[x] = E::kMaskWord;
#pragma unroll
        for (int x = 0; x < 16; ++x) rq[x] = INT32_MIN;
        auto take = [&](const uint32_t (&w)[8], int cls) -> int32_t {
            int32_t vm;
            if constexpr (BF16) {
                const uint32_t pa = max_s16x2(max_s16x2(w[0], w[2]), max_s16x2(w[4], w[6]));
                const uint32_t pb = max_s16x2(max_s16x2(w[1], w[3]), max_s16x2(w[5], w[7]));
                rp[cls * 2] = max_s16x2(rp[cls * 2], pa);
                rp[cls * 2 + 1] = max_s16x2(rp[cls * 2 + 1], pb);
                const uint32_t mm = max_s16x2(pa, pb);
                vm = max(E::pack_lo(mm), E::pack_hi(mm));
            } else {
                int32_t m4[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    m4[jj] = max((int32_t)w[jj], (int32_t)w[jj + 4]);
                    rq[cls * 4 + jj] = max(rq[cls * 4 + jj], m4[jj]);
                }
                vm = max(max(m4[0], m4[1]), max(m4[2], m4[3])) >> 16;
            }
            return vm;
        };
        // The same on raw bits (interior chunks, bf16): a subset's largest key
        // is its raw signed maximum when that is non-negative, else the key of
        // its raw signed minimum (a negative value's magnitude grows with its
        // raw integer, so the most negative raw value is the largest float),
        // with the low 15 bits flipped.
        auto take_raw = [&](const uint32_t (&w)[8], int cls) -> int32_t {
            if constexpr (BF16) {
                const uint32_t ax = max_s16x2(max_s16x2(w[0], w[2]), max_s16x2(w[4], w[6]));
                const uint32_t an = min_s16x2(min_s16x2(w[0], w[2]), min_s16x2(w[4], w[6]));
                const uint32_t bx = max_s16x2(max_s16x2(w[1], w[3]), max_s16x2(w[5], w[7]));
                const uint32_t bn = min_s16x2(min_s16x2(w[1], w[3]), min_s16x2(w[5], w[7]));
                // 0xFFFF in each half whose raw maximum is negative
                const uint32_t ma = sign_mask16(ax), mb = sign_mask16(bx);
                const uint32_t pa = (ax & ~ma) | ((an ^ 0x7FFF7FFFu) & ma);
                const uint32_t pb = (bx & ~mb) | ((bn ^ 0x7FFF7FFFu) & mb);
                rp[cls * 2] = max_s16x2(rp[cls * 2], pa);
                rp[cls * 2 + 1] = max_s16x2(rp[cls * 2 + 1], pb);
                const uint32_t mm = max_s16x2(pa, pb);
                return max(E::pack_lo(mm), E::pack_hi(mm));
            } else {
                uint32_t k[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) k[x] = w[x];
                chunk_to_keys<BF16>(k);
                return take(k, cls);
            }
        };
        auto store_vmax = [&](int i, int32_t v0, int32_t v1) {
            sm.a.vmax2[i][lane] = ((uint32_t)v0 & 0xFFFFu) | ((uint32_t)v1 << 16);
        };
        // Step 0 splits each chunk finer, into 8 subsets spread over the
        // four classes, so that a short row (a few chunks) still has at least
        // K' representatives and a tight theta.
        auto take_first = [&](const uint32_t (&w)[8], int c) -> int32_t {
            int32_t vm;
            if constexpr (BF16) {
                const uint32_t a0 = max_s16x2(w[0], w[4]), a1 = max_s16x2(w[2], w[6]);
                const uint32_t b0 = max_s16x2(w[1], w[5]), b1 = max_s16x2(w[3], w[7]);
                rp[2 * c] = max_s16x2(rp[2 * c], a0);
                rp[2 * c + 1] = max_s16x2(rp[2 * c + 1], b0);
                rp[2 * c + 4] = max_s16x2(rp[2 * c + 4], a1);
                rp[2 * c + 5] = max_s16x2(rp[2 * c + 5], b1);
                const uint32_t mm = max_s16x2(max_s16x2(a0, a1), max_s16x2(b0, b1));
                vm = max(E::pack_lo(mm), E::pack_hi(mm));
            } else {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    rq[c * 4 + jj] = max(rq[c * 4 + jj], (int32_t)w[jj]);
                    rq[(c + 2) * 4 + jj] = max(rq[(c + 2) * 4 + jj], (int32_t)w[jj + 4]);
                }
                int32_t m = (int32_t)w[0];
#pragma unroll
                for (int jj = 1; jj < 8; ++jj) m = max(m, (int32_t)w[jj]);
                vm = m >> 16;
            }
            return vm;
        };
        const int nsteps = need ? (nchunk + 3) >> 2 : 0;
        // step 0 and the last step hold the row's edge chunks: masked loads
        auto edge_step = [&](int i, int cls0) {
            int32_t vm[2] = {-32768, -32768};
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int k = 4 * i + 2 * s + c;
                if (k < nchunk) {
                    uint32_t w[8];
                    pair_load_edge<BF16>(P, k, c0, base_id, r.lo, r.hi, row_ptr, w);
                    vm[c] = i == 0 ? take_first(w, c) : take(w, cls0 + c);
                }
            }
            store_vmax(i, vm[0], vm[1]);
        };
        if (nsteps > 0) edge_step(0, 0);
        // interior steps 1 .. i_last hold chunks <= nchunk - 2 only; the next
        // step's two chunks are loaded while the current one is reduced
        const int i_last = nsteps >= 2 ? (nchunk - 5) / 4 : 0;
        if (i_last >= 1) {
            // ping-pong between buffers A and B: odd steps in A, even in B
            uint32_t a0[8], a1[8], b0[8], b1[8];
            uintptr_t ad = c0 + ((uintptr_t)(4 + 2 * s) << 5);
            ld32(ad, a0);
            ld32(ad + 32, a1);
            for (int i = 1; i <= i_last; i += 2) {
                if (i < i_last) {
                    ld32(ad + 128, b0);
                    ld32(ad + 160, b1);
                }
                const int32_t va0 = take_raw(a0, 0);
                store_vmax(i, va0, take_raw(a1, 1));
                if (i < i_last) {
                    if (i + 1 < i_last) {
                        ld32(ad + 256, a0);
                        ld32(ad + 288, a1);
                    }
                    const int32_t vb0 = take_raw(b0, 2);
                    store_vmax(i + 1, vb0, take_raw(b1, 3));
                }
                ad += 256;
            }
        }
        if (nsteps >= 2) edge_step(nsteps - 1, 2);

        // ---- theta: the K'-th largest of the row's 32 representatives (distinct
        // elements), a lower bound on the K'-th best score ----
        // bitonic sort of the pair's 32 representatives; the K'-th largest is
        // position K' - 1.  A row with fewer than K' representatives gets the
        // smallest key: every element of [lo, hi) is then a candidate.
        const int want = max(r.kp - 1, 0);
        int32_t theta;
        if constexpr (SMALLK && BF16) {
            // K' <= 16: the top 16 suffice; bf16 representatives stay packed
            packed_pair_top16_desc<true>(rp);
            const uint32_t wv = pick(rp, want & 7);
            theta = (int32_t)(int16_t)(uint16_t)(want < 8 ? wv : (wv >> 16));
        } else {
            int32_t rep[16];
            if constexpr (BF16) {
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    rep[2 * x] = E::pack_lo(rp[x]);
                    rep[2 * x + 1] = E::pack_hi(rp[x]);
                }
            } else {
#pragma unroll
                for (int x = 0; x < 16; ++x) rep[x] = rq[x];
            }
            if constexpr (SMALLK) {
                // K' <= 16: the top 16 suffice, in lane 0
                pair_top16_desc<int32_t>(rep);
                theta = __shfl_sync(kFull, pick(rep, want), lane & ~1);
            } else {
                pair_sort32_desc<int32_t>(rep, s);
                const int32_t mine = pick(rep, want & 15);
                const int32_t other = __shfl_xor_sync(kFull, mine, 1);
                theta = ((want < 16) == (s == 0)) ? mine : other;
            }
        }
        if (s == 0) {
            sm.ccount[p] = 0;
            sm.ovf[p] = 0;
            PairRowDesc d;
            d.c0 = c0;
            d.row_ptr = reinterpret_cast<uintptr_t>(row_ptr);
            d.base_id = base_id;
            d.lo = r.lo;
            d.hi = r.hi;
            d.theta = theta;
            d.nchunk = nchunk;
            d.inside = (c0 >= P.buf_lo && c0 + ((uintptr_t)nchunk << 5) <= P.buf_hi) ? 1 : 0;
            sm.desc[p] = d;
        }
        const int32_t th16 = BF16 ? theta : (theta >> 16);

        // ---- queue the chunks that can hold candidates ----
        // lane-local entry j holds chunk 4 (j >> 1) + 2 s + (j & 1); the
        // entries below jmax exist.  Eight chunk maxima per packed compare.
        const int jmax = need ? 2 * (nchunk >> 2) + min(max((nchunk & 3) - 2 * s, 0), 2) : 0;
        unsigned long long hot = 0;
        for (int i0 = 0; i0 < jmax; i0 += 8) {
            const uint32_t wv[4] = {sm.a.vmax2[i0 / 2][lane], sm.a.vmax2[i0 / 2 + 1][lane],
                                    sm.a.vmax2[i0 / 2 + 2][lane], sm.a.vmax2[i0 / 2 + 3][lane]};
            const uint32_t bits = th16 == -32768 ? 0xFFu : ge_bits16<4>(wv, th16);
            hot |= (unsigned long long)bits << i0;
        }
        hot &= (1ull << jmax) - 1ull;
        int qtotal;
        int qpos = warp_excl_scan(__popcll(hot), lane, qtotal);
        // entry (p << 8 | k), k = 4 (j >> 1) + 2 s + (j & 1) = 2 j - (j & 1) + 2 s;
        // entries j >= 32 exist only for rows of more than 64 chunks
        const int ebase = (p << 8) | (2 * s);
        uint32_t hlo = (uint32_t)hot;
        while (hlo) {
            const int j = __ffs(hlo) - 1;
            hlo &= hlo - 1;
            sm.q.queue[qpos++] = (uint16_t)(ebase + 2 * j - (j & 1));
        }
        uint32_t hhi = (uint32_t)(hot >> 32);
        while (hhi) {
            const int j = 32 + __ffs(hhi) - 1;
            hhi &= hhi - 1;
            sm.q.queue[qpos++] = (uint16_t)(ebase + 2 * j - (j & 1));
        }
        const int qn = qtotal;
        __syncwarp();   // vmax is dead from here on; its space holds the scratch

        // ---- candidates from the queued chunks, 32 at a time ----
        // Every chunk is loaded whole (it lies inside the score buffer unless
        // the row's edges cross the buffer's ends, which the edge loader
        // handles); ids outside [lo, hi) are cut by a range mask; keys >=
        // theta are found with packed compares and emitted through a per-lane
        // scratch.
        for (int base = 0; base < qn; base += 32) {
            const int e = base + lane;
            if (e < qn) {
                const int ent = sm.q.queue[e];
                const int pp = ent >> 8;
                const int k = ent & 0xFF;
                const PairRowDesc d = sm.desc[pp];
                uint32_t w[8];
                const uintptr_t addr = (uintptr_t)d.c0 + ((uintptr_t)k << 5);
                if (d.inside || (addr >= P.buf_lo && addr + 32 <= P.buf_hi)) {
                    ld32(addr, w);
                    // against theta >= 0, raw signed order is key order
                    if (d.theta < 0) chunk_to_keys<BF16>(w);
                } else {
                    pair_load_edge<BF16>(P, k, (uintptr_t)d.c0, d.base_id, d.lo, d.hi,
                                         reinterpret_cast<const char*>(d.row_ptr), w);
                    if (d.theta >= 0) chunk_to_keys<BF16>(w);  // back to raw bits
                }
                const int first_id = d.base_id + k * CE;
                // bf16 masks use the ge_bits16_perm order
                uint32_t m = BF16 ? 0xFFFFu : 0xFFu;
                if (k == 0 || k == d.nchunk - 1) {
                    // an edge chunk: cut ids outside [lo, hi)
                    const int lo_e = min(max(d.lo - first_id, 0), CE);
                    const int hi_e = min(max(d.hi - first_id, 0), CE);
                    if constexpr (BF16) {
                        auto range = [](int a, int b) { return ((1u << b) - 1u) & ~((1u << a) - 1u); };
                        m = range((lo_e + 1) >> 1, (hi_e + 1) >> 1) |
                            (range(lo_e >> 1, hi_e >> 1) << 8);
                    } else {
                        m = ((1u << hi_e) - 1u) & ~((1u << lo_e) - 1u);
                    }
                }
                if (d.theta != kKeyMin) {
                    if constexpr (BF16) {
                        m &= ge_bits16_perm(w, d.theta);
                    } else {
                        uint32_t bits = 0;
#pragma unroll
                        for (int x = 0; x < 8; ++x) bits |= ((int32_t)w[x] >= d.theta ? 1u : 0u) << x;
                        m &= bits;
                    }
                }
                const int nc = __popc(m);
                if (nc) {
                    int pos = atomicAdd(&sm.ccount[pp], nc);
                    if (pos + nc <= kPairCand) {
                        uint32_t* scr = sm.a.scratch[lane];
#pragma unroll
                        for (int x = 0; x < 8; ++x) scr[x] = w[x];
                        while (m) {
                            const int b = __ffs(m) - 1;
                            m &= m - 1;
                            const int x = BF16 ? perm_elem(b) : b;
                            uint32_t ukey;
                            if constexpr (BF16)
                                ukey = ((uint32_t)reinterpret_cast<const uint16_t*>(scr)[x]) ^ kFlip;
                            else
                                ukey = scr[x] ^ kFlip;
                            sm.cand[pp][pos++] = make_ck<CK>(ukey, first_id + x);
                        }
                    } else {
                        sm.ovf[pp] = 1;
                    }
                }
            }
        }
        __syncwarp();

        {
            // the row's geometry again from its page count (passed through an
            // opaque move, so that the compiler recomputes it rather than
            // holding it in registers through the candidate phase)
            int32_t m2;
            asm volatile("mov.b32 %0, %1;" : "=r"(m2) : "r"(cur_meta));
            RowInfo r2{};
            r2.all = true;
            if (active) r2 = row_info_from<FM>(a, row, m2);
            r = r2;
        }
        // ---- exact select: sort the row's candidates, keep the first K' ----
        const bool ovf = sm.ovf[p] != 0;
        const int cn = min(sm.ccount[p], kPairCand);
        const bool sel_ok = need && !ovf;
        CK x[16];
        {
            // this lane's 16 list positions with vector loads, then the mask
            const uint4* src = reinterpret_cast<const uint4*>(&sm.cand[p][s * 16]);
            constexpr int kPer = 16 / sizeof(CK);   // composite keys per 16 bytes
#pragma unroll
            for (int v = 0; v < 16 / kPer; ++v) {
                const uint4 q4 = src[v];
                const CK* e = reinterpret_cast<const CK*>(&q4);
#pragma unroll
                for (int t = 0; t < kPer; ++t) x[v * kPer + t] = e[t];
            }
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (!(sel_ok && s * 16 + u < cn)) x[u] = (CK)0;
        }
        if constexpr (SMALLK)
            pair_top16_desc<CK>(x);
        else
            pair_sort32_desc<CK>(x, s);
        __syncwarp();
        if constexpr (SMALLK) {
            // K' <= 16: the kept positions are lane 0's registers.  Their ids
            // (< 2^16 on this path) are sorted as 0xFFFF - id, two per word.
            uint32_t yp[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const uint32_t lo = (s == 0 && u < r.kp)
                                        ? 0xFFFFu - (uint32_t)(kLowMax - ck_low(x[u])) : 0u;
                const uint32_t hi = (s == 0 && u + 8 < r.kp)
                                        ? 0xFFFFu - (uint32_t)(kLowMax - ck_low(x[u + 8])) : 0u;
                yp[u] = lo | (hi << 16);
            }
            packed_sort16_desc<false>(yp);
            if (sel_ok && s == 0) {
                // id = 0xFFFF - value = the value's complement; positions >= K'
                // are never read
                int4* dst = reinterpret_cast<int4*>(sm.q.sorted[p]);
#pragma unroll
                for (int v = 0; v < 2; ++v) {
                    dst[v] = make_int4((int32_t)(~yp[4 * v] & 0xFFFFu), (int32_t)(~yp[4 * v + 1] & 0xFFFFu),
                                       (int32_t)(~yp[4 * v + 2] & 0xFFFFu),
                                       (int32_t)(~yp[4 * v + 3] & 0xFFFFu));
                    dst[v + 2] = make_int4((int32_t)(~yp[4 * v] >> 16), (int32_t)(~yp[4 * v + 1] >> 16),
                                           (int32_t)(~yp[4 * v + 2] >> 16),
                                           (int32_t)(~yp[4 * v + 3] >> 16));
                }
            }
        } else {
            uint32_t y[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) y[u] = (s * 16 + u < r.kp) ? ck_low(x[u]) : 0u;
            pair_sort32_desc<uint32_t>(y, s);
            if (sel_ok) {
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    if (s * 16 + u < r.kp) sm.q.sorted[p][s * 16 + u] = (int32_t)(kLowMax - y[u]);
            }
        }
        __syncwarp();

        // ---- outputs ----
        group_write_outputs<2, FM>(P, row, r, r.all, sm.q.sorted[p], s,
                                   active && !longr && (!need || !ovf));

        // ---- rows whose candidates overflowed: the whole warp redoes them ----
        unsigned fb = __ballot_sync(kFull, s == 0 && need && ovf);
        __syncwarp();
        while (fb) {
            const int bit = __ffs(fb) - 1;
            fb &= fb - 1;
            const int64_t frow = (int64_t)it * kPairRows + (bit >> 1);
            uint32_t* s_keys = reinterpret_cast<uint32_t*>(&sm);
            warp_item<BF16, 4, 2>(P, frow, 0, s_keys, reinterpret_cast<int32_t*>(s_keys + P.cap),
                                  lane);
            __syncwarp();
        }
        __syncwarp();
    }
}

// ===========================================================================
// Octet path: 8 lanes per row, 4 rows per warp, for 32 < topk <= 64.
//
// At topk 64 nearly every 32-byte chunk of a long row holds one of the K'
// best elements, so the pair path's hot-chunk queue would reload almost the
// whole row, and a lane pair's 32 representatives give no threshold for
// K' > 32.  Here the 8 lanes of a row:
//  1. stream its non-forced range in 32-byte chunks (256 contiguous bytes per
//     row per step) and keep, for each of the 16 element positions of a
//     chunk, the largest key seen there: 16 representatives per lane and up
//     to 128 per row, each the maximum of distinct elements.  Chunks are
//     reduced on raw bits (a raw maximum and minimum per position, turned
//     into the key maximum once at the end).  The two edge chunks are left
//     out: a row that needs a threshold has at least 9 chunks, so lanes 1-7
//     hold interior ones and each quad keeps at least 32 representatives.
//  2. theta: each quad of lanes (64 representatives) finds its 32nd largest
//     representative with packed 16-bit bitonic networks (each lane sorts its
//     16, lane pairs merge into a sorted 32, the top 32 of the quad's two
//     pairs are their pairwise maxima); theta is the smaller of the two
//     quads' values.  At least 64 >= K' representatives, distinct elements,
//     reach theta, so it is a lower bound on the K'-th best non-forced score.
//     fp32 rows use the top 16 bits of their keys for this step.
//  3. candidates: the chunks are read again in order (L2 hits: the row was
//     prefetched to L2 when its item began), and the elements >= theta are
//     appended to a 128-entry list in id order, a segmented scan over the 8
//     lanes giving each lane its place.  Rows of at most 128 non-forced
//     blocks skip steps 1-2: every element is a candidate.
//  4. kappa, the K'-th largest candidate key, by a binary search over
//     [theta, largest candidate] with the candidates spread 16 per lane.  The
//     candidates above kappa are kept, and of those equal to it the first in
//     id order, as many as K' still needs; the kept ids, in id order, are
//     compacted into the sorted list.
//  5. outputs as on the other paths (8 slots per lane at topk 64).
// A row whose candidates overflow the list (about 1 row in 1000 on N(0,1)
// scores, in a CPU model of the long-context input) is redone by the whole
// warp on the warp path.
// ===========================================================================

// Exclusive sum of x over the 8 lanes of this lane's row; `total` gets the
// row's sum.  Every lane of the warp calls this.
__device__ __forceinline__ int oct_excl_scan(int x, int q, int& total) {
    int incl = x;
#pragma unroll
    for (int d = 1; d < kOctLanes; d <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, d);
        if (q >= d) incl += y;
    }
    total = __shfl_sync(kFull, incl, (int)(threadIdx.x & 31) | (kOctLanes - 1));
    return incl - x;
}

__device__ __forceinline__ int oct_sum(int x) {
    x += __shfl_xor_sync(kFull, x, 1);
    x += __shfl_xor_sync(kFull, x, 2);
    x += __shfl_xor_sync(kFull, x, 4);
    return x;
}

// Step 2: from the lane's 16 representatives (signed 16-bit keys, packed two
// per word), the smaller of the row's two quad values (each the 32nd largest
// of a quad's 64 representatives).  Every lane of the warp calls this.
__device__ __forceinline__ int32_t oct_theta(uint32_t (&rp)[8], int q) {
    packed_sort16_desc<true>(rp);
    // lane pairs: the even lane keeps the top 16 of the pair's 32, the odd
    // lane the bottom 16 (each bitonic), then both are sorted; word i of a
    // lane holds its positions i (low half) and i + 8 (high half), and the
    // partner's list reversed is its word 7 - i with the halves swapped
    uint32_t y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __shfl_xor_sync(kFull, rp[7 - i], 1);
    const bool top = (q & 1) == 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t b = __byte_perm(y[i], 0, 0x1032);
        rp[i] = top ? hmax<true>(rp[i], b) : hmin<true>(rp[i], b);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) rp[i] = hsplit<true>(rp[i]);
    hclean8_desc<true>(rp);
    // quads: with P0 the sorted 32 of lanes 0-1 and P1 that of lanes 2-3,
    // max(P0[r], P1[31 - r]) over r are the quad's top 32; lane q meets lane
    // q ^ 3's list reversed.  Their minimum is the quad's 32nd largest.
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __shfl_xor_sync(kFull, rp[7 - i], 3);
    uint32_t mn = 0x7FFF7FFFu;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        mn = hmin<true>(mn, hmax<true>(rp[i], __byte_perm(y[i], 0, 0x1032)));
    int32_t m = min((int32_t)(int16_t)(uint16_t)mn, (int32_t)(int16_t)(uint16_t)(mn >> 16));
    m = min(m, __shfl_xor_sync(kFull, m, 1));
    m = min(m, __shfl_xor_sync(kFull, m, 4));
    return m;
}

// TAIL: rows over 2 KB are listed for the wide path (buffers wider than
// 2 KB); without it the kernel has none of that code.
template <bool BF16, int FM, bool TAIL>
__global__ void __launch_bounds__(kOctWarps * 32,
                                  FM == kFusedNo && BF16 ? kOctCtasSelect : kOctCtas)
    octet_select_kernel(const KernelParams P) {
    using E = Elem<BF16>;
    constexpr int S = E::kBytes;
    constexpr int CE = 32 / S;                      // elements per 32-byte chunk
    constexpr int32_t kKeyMin = BF16 ? -32768 : INT32_MIN;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int g = lane >> 3;   // row of the warp's item
    const int q = lane & 7;    // lane within the row
    OctSmem& sm = *reinterpret_cast<OctSmem*>(smem_raw + (size_t)warp * sizeof(OctSmem));
    const SelectArgs& a = P.a;
    const int64_t nitems = (P.rows + kOctRows - 1) / kOctRows;
    const int64_t stride = (int64_t)gridDim.x * kOctWarps;

    for (int64_t it = (int64_t)blockIdx.x * kOctWarps + warp; it < nitems; it += stride) {
        const int64_t row = it * kOctRows + g;
        const bool active = row < P.rows;
        RowInfo r{};
        r.all = true;
        if (active) r = row_info_from<FM>(a, row, row_meta<FM>(a, row));
        // a row whose range exceeds 2 KB (a wider buffer) goes to the list of
        // the second, wide-path launch
        const bool longr = TAIL && active && r.need && (int64_t)(r.hi - r.lo) * S > kGroupMaxBytes;
        if (longr && q == 0) P.long_list[atomicAdd(P.long_count, 1u)] = (int32_t)row;
        const bool need = active && r.need && !longr;

        // ---- geometry of the non-forced range [lo, hi), 32-byte chunks ----
        const char* row_ptr = nullptr;
        uintptr_t c0 = 0;
        int nchunk = 0, base_id = 0;
        if (need) {
            row_ptr = reinterpret_cast<const char*>(a.scores) +
                      ((int64_t)r.t * a.token_stride + (int64_t)r.h * a.head_stride) * S;
            const uintptr_t a_lo = reinterpret_cast<uintptr_t>(row_ptr) + (uintptr_t)r.lo * S;
            const uintptr_t a_hi = reinterpret_cast<uintptr_t>(row_ptr) + (uintptr_t)r.hi * S;
            c0 = a_lo & ~(uintptr_t)31;
            nchunk = (int)((a_hi - c0 + 31) >> 5);
            base_id = r.lo - (int)((a_lo - c0) / S);
            if (q == 0) {
                const uintptr_t plo = c0 < P.buf_lo ? (P.buf_lo + 15) & ~(uintptr_t)15 : c0;
                uintptr_t phi = c0 + ((uintptr_t)nchunk << 5);
                if (phi > P.buf_hi) phi = P.buf_hi & ~(uintptr_t)15;
                if (phi > plo) prefetch_l2(plo, (uint32_t)(phi - plo));
            }
        }
        // rows of more than kOctCand non-forced blocks need a threshold
        const bool full = need && (r.hi - r.lo) > kOctCand;

        // ---- step 1: 16 representatives per lane (packed 16-bit keys) ----
        uint32_t rp[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) rp[x] = 0x80008000u;
        if (full) {
            // full rows have at least 129 non-forced blocks: every lane owns a chunk
            if constexpr (BF16) {
                uint32_t rmx[8], rmn[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    rmx[x] = 0x80008000u;
                    rmn[x] = 0x7FFF7FFFu;
                }
                auto fold = [&](const uint32_t (&w)[8]) {
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        rmx[x] = max_s16x2(rmx[x], w[x]);
                        rmn[x] = min_s16x2(rmn[x], w[x]);
                    }
                };
                // interior chunks k = q + 8 i, 1 <= k <= nchunk - 2, two loads
                // in flight; the edge chunks (0 and nchunk - 1) are left out
                const int klast = nchunk - 2;
                int k = q == 0 ? kOctLanes : q;
                const bool any_interior = k <= klast;
                for (; k + kOctLanes <= klast; k += 2 * kOctLanes) {
                    uint32_t w0[8], w1[8];
                    ld32(c0 + ((uintptr_t)k << 5), w0);
                    ld32(c0 + ((uintptr_t)(k + kOctLanes) << 5), w1);
                    fold(w0);
                    fold(w1);
                }
                if (k <= klast) {
                    uint32_t w0[8];
                    ld32(c0 + ((uintptr_t)k << 5), w0);
                    fold(w0);
                }
                if (any_interior) {
                    // a position's largest key: its raw maximum when that is
                    // non-negative, else the key of its raw minimum
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        const uint32_t mneg = sign_mask16(rmx[x]);
                        const uint32_t km = (rmx[x] & ~mneg) | ((rmn[x] ^ 0x7FFF7FFFu) & mneg);
                        rp[x] = max_s16x2(rp[x], km);
                    }
                }
            } else {
                // fp32: 8 positions per chunk, two sets by the lane's chunk
                // parity, so a lane with two or more chunks has 16
                // representatives; packed as the top 16 bits of the keys
                int32_t ra[8], rb[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) ra[x] = rb[x] = INT32_MIN;
                // interior chunks only, as for bf16
                for (int k = q; k < nchunk; k += 2 * kOctLanes) {
                    uint32_t w0[8], w1[8];
                    const bool one = k != 0 && k != nchunk - 1;
                    const int k1 = k + kOctLanes;
                    const bool two = k1 < nchunk - 1;
                    if (one) ld32(c0 + ((uintptr_t)k << 5), w0);
                    if (two) ld32(c0 + ((uintptr_t)k1 << 5), w1);
                    if (one) {
                        chunk_to_keys<false>(w0);
#pragma unroll
                        for (int x = 0; x < 8; ++x) ra[x] = max(ra[x], (int32_t)w0[x]);
                    }
                    if (two) {
                        chunk_to_keys<false>(w1);
#pragma unroll
                        for (int x = 0; x < 8; ++x) rb[x] = max(rb[x], (int32_t)w1[x]);
                    }
                }
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    rp[x] = ((uint32_t)ra[2 * x] >> 16) | ((uint32_t)ra[2 * x + 1] & 0xFFFF0000u);
                    rp[x + 4] = ((uint32_t)rb[2 * x] >> 16) | ((uint32_t)rb[2 * x + 1] & 0xFFFF0000u);
                }
            }
        }

        // ---- step 2: theta (every lane takes part in the networks) ----
        const int32_t th16 = oct_theta(rp, q);
        int32_t theta = kKeyMin;
        if (full) theta = BF16 ? th16 : (int32_t)((uint32_t)th16 << 16);

        // ---- step 3: candidates >= theta, in id order ----
        const int my_steps = need ? (nchunk - q + kOctLanes - 1) / kOctLanes : 0;
        const int steps = __reduce_max_sync(kFull, (unsigned)my_steps);
        const bool raw_ok = theta >= 0;   // raw signed order is key order against it
        int cbase = 0;
        // the next step's chunk is loaded while this one is processed; an
        // edge chunk is loaded whole when it lies inside the score buffer (its
        // ids outside [lo, hi) are cut by the range mask below)
        uint32_t nx[8];
        auto plain = [&](int k) {
            const uintptr_t addr = c0 + ((uintptr_t)k << 5);
            return (k != 0 && k != nchunk - 1) || (addr >= P.buf_lo && addr + 32 <= P.buf_hi);
        };
        auto issue = [&](int st) {
            const int k = q + kOctLanes * st;
            if (k < nchunk && plain(k)) ld32(c0 + ((uintptr_t)k << 5), nx);
        };
        issue(0);
        for (int st = 0; st < steps; ++st) {
            const int k = q + kOctLanes * st;
            const bool has = k < nchunk;
            uint32_t w[8];
            uint32_t m = 0;
            if (has) {
                if (!plain(k)) {
                    // masked keys, which compare like raw bits against theta >= 0
                    pair_load_edge<BF16>(P, k, c0, base_id, r.lo, r.hi, row_ptr, w);
                } else {
#pragma unroll
                    for (int x = 0; x < 8; ++x) w[x] = nx[x];
                    if (!raw_ok) chunk_to_keys<BF16>(w);
                }
            }
            issue(st + 1);
            if (has) {
                const bool edge = k == 0 || k == nchunk - 1;
                if (theta == kKeyMin) {
                    m = BF16 ? 0xFFFFu : 0xFFu;
                } else if constexpr (BF16) {
                    m = ge_bits16<8>(w, theta);
                } else {
#pragma unroll
                    for (int x = 0; x < 8; ++x) m |= ((int32_t)w[x] >= theta ? 1u : 0u) << x;
                }
                if (edge) {
                    const int first_id = base_id + k * CE;
                    const int lo_e = min(max(r.lo - first_id, 0), CE);
                    const int hi_e = min(max(r.hi - first_id, 0), CE);
                    m &= ((1u << hi_e) - 1u) & ~((1u << lo_e) - 1u);
                }
            }
            int tot;
            const int off = oct_excl_scan(__popc(m), q, tot);
            if (m) {
                uint32_t* scr = sm.scratch[lane];
#pragma unroll
                for (int x = 0; x < 8; ++x) scr[x] = w[x];
                const int first_id = base_id + k * CE;
                int pos = cbase + off;
                while (m) {
                    const int e = __ffs(m) - 1;
                    m &= m - 1;
                    if (pos < kOctCand) {
                        if constexpr (BF16)
                            sm.ckey16[g][pos] = reinterpret_cast<const int16_t*>(scr)[e];
                        else
                            sm.ckey[g][pos] = (int32_t)scr[e];
                        sm.cid[g][pos] = (uint16_t)(first_id + e);
                    }
                    ++pos;
                }
            }
            cbase += tot;
        }
        const bool ovf = cbase > kOctCand;
        __syncwarp();

        // ---- step 4: kappa, the K'-th largest candidate key ----
        // A binary search over [theta, largest candidate]: count(>= lo) >= K'
        // > count(>= hi) = cnt_hi throughout.  The lane's list positions
        // 16 q .. 16 q + 15 past the count c are masked out.
        const bool sel_ok = need && !ovf;
        const int c = min(cbase, kOctCand);
        const int nvalid = sel_ok ? min(max(c - 16 * q, 0), 16) : 0;
        const uint32_t valid = (1u << nvalid) - 1u;
        const int kp = r.kp;
        uint32_t gtm = 0, eqm = 0;
        int cnt_hi = 0;
        if constexpr (BF16) {
            // 16 keys per lane, two per word; padding holds -32768, which no
            // searched threshold (> lo >= -32768) counts
            uint32_t kw[8];
            {
                const uint4* src = reinterpret_cast<const uint4*>(&sm.ckey16[g][16 * q]);
                const uint4 v0 = src[0], v1 = src[1];
                kw[0] = v0.x; kw[1] = v0.y; kw[2] = v0.z; kw[3] = v0.w;
                kw[4] = v1.x; kw[5] = v1.y; kw[6] = v1.z; kw[7] = v1.w;
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    const uint32_t keep = ((valid >> (2 * x)) & 1u ? 0x0000FFFFu : 0u) |
                                          ((valid >> (2 * x + 1)) & 1u ? 0xFFFF0000u : 0u);
                    kw[x] = (kw[x] & keep) | (0x80008000u & ~keep);
                }
            }
            uint32_t mw = kw[0];
#pragma unroll
            for (int x = 1; x < 8; ++x) mw = max_s16x2(mw, kw[x]);
            int32_t mx = max((int32_t)(int16_t)(uint16_t)mw, (int32_t)(int16_t)(uint16_t)(mw >> 16));
            mx = max(mx, __shfl_xor_sync(kFull, mx, 1));
            mx = max(mx, __shfl_xor_sync(kFull, mx, 2));
            mx = max(mx, __shfl_xor_sync(kFull, mx, 4));
            int32_t lo = theta, hi = mx + 1;
            if (!sel_ok) hi = lo + 1;
            while (__any_sync(kFull, hi - lo > 1)) {
                const int32_t mid = (lo + hi) >> 1;
                const uint32_t t2 = ((uint32_t)(mid - 1) & 0xFFFFu) * 0x10001u;
                uint32_t sacc = 0;
#pragma unroll
                for (int x = 0; x < 8; ++x) sacc += min_u16x2(max_s16x2(kw[x], t2) ^ t2, 0x00010001u);
                const int cnt = oct_sum((int)((sacc & 0xFFFFu) + (sacc >> 16)));
                if (hi - lo > 1) {
                    if (cnt >= kp) {
                        lo = mid;
                    } else {
                        hi = mid;
                        cnt_hi = cnt;
                    }
                }
            }
            // kappa = lo: keep every candidate above it and the first
            // (K' - count above) of those equal to it, in id order
            if (sel_ok) {
                gtm = ge_bits16<8>(kw, lo + 1) & valid;
                eqm = (lo == kKeyMin ? valid : ge_bits16<8>(kw, lo) & valid) & ~gtm;
            }
        } else {
            int32_t kk[16];
            {
                const int4* src = reinterpret_cast<const int4*>(&sm.ckey[g][16 * q]);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int4 t4 = src[v];
                    kk[4 * v] = t4.x;
                    kk[4 * v + 1] = t4.y;
                    kk[4 * v + 2] = t4.z;
                    kk[4 * v + 3] = t4.w;
                }
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (!((valid >> e) & 1u)) kk[e] = INT32_MIN;
            }
            int32_t mx = INT32_MIN;
#pragma unroll
            for (int e = 0; e < 16; ++e) mx = max(mx, kk[e]);
            mx = max(mx, __shfl_xor_sync(kFull, mx, 1));
            mx = max(mx, __shfl_xor_sync(kFull, mx, 2));
            mx = max(mx, __shfl_xor_sync(kFull, mx, 4));
            // the padding (INT32_MIN) is never counted because mid > lo
            int64_t lo = theta, hi = (int64_t)mx + 1;
            if (!sel_ok) hi = lo + 1;
            while (__any_sync(kFull, hi - lo > 1)) {
                const int64_t mid = lo + ((hi - lo) >> 1);
                const int32_t t = (int32_t)mid;
                int cnt = 0;
#pragma unroll
                for (int e = 0; e < 16; ++e) cnt += kk[e] >= t ? 1 : 0;
                cnt = oct_sum(cnt);
                if (hi - lo > 1) {
                    if (cnt >= kp) {
                        lo = mid;
                    } else {
                        hi = mid;
                        cnt_hi = cnt;
                    }
                }
            }
            const int32_t kappa = (int32_t)lo;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const bool vd = (valid >> e) & 1u;
                if (vd && kk[e] > kappa) gtm |= 1u << e;
                if (vd && kk[e] == kappa) eqm |= 1u << e;
            }
        }
        int tall;
        const int tb = oct_excl_scan(__popc(eqm), q, tall);
        const int allowed = min(max(kp - cnt_hi - tb, 0), __popc(eqm));
        uint32_t rest = eqm;
        for (int i = 0; i < allowed; ++i) rest &= rest - 1;
        uint32_t selm = gtm | (eqm & ~rest);
        int stot;
        int o = oct_excl_scan(__popc(selm), q, stot);
        while (selm) {
            const int e = __ffs(selm) - 1;
            selm &= selm - 1;
            sm.sorted[g][o++] = sm.cid[g][16 * q + e];
        }
        __syncwarp();

        // ---- step 5: outputs ----
        group_write_outputs<kOctLanes, FM>(P, row, r, r.all, sm.sorted[g], q,
                                           active && !longr && (!need || !ovf));

        // ---- rows whose candidates overflowed: the whole warp redoes them ----
        unsigned fb = __ballot_sync(kFull, q == 0 && need && ovf);
        __syncwarp();
        while (fb) {
            const int bit = __ffs(fb) - 1;
            fb &= fb - 1;
            const int64_t frow = it * kOctRows + (bit >> 3);
            uint32_t* s_keys = reinterpret_cast<uint32_t*>(&sm);
            warp_item<BF16, 4, 2>(P, frow, 0, s_keys, reinterpret_cast<int32_t*>(s_keys + P.cap),
                                  lane);
            __syncwarp();
        }
        __syncwarp();
    }
}

template <bool BF16>
cudaError_t launch_octet(const KernelParams& P, const bsa_launch_policy_t& pol, cudaStream_t st) {
    auto kern = P.a.fused ? octet_select_kernel<BF16, kFusedYes, false>
                          : octet_select_kernel<BF16, kFusedNo, false>;
    if (P.long_list != nullptr)
        kern = P.a.fused ? octet_select_kernel<BF16, kFusedYes, true>
                         : octet_select_kernel<BF16, kFusedNo, true>;
    if (pol.smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             pol.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    kern<<<pol.grid, kOctWarps * 32, pol.smem_bytes, st>>>(P);
    return cudaGetLastError();
}

// ===========================================================================
// Wide path: one warp per row, for rows of a buffer wider than 2 KB (bf16
// capacities above 1024 tiles, fp32 above 512, up to the 8192-tile
// capture-time capacity) and topk <= 64.  The octet path's steps with all 32
// lanes on one row (fp32 as on the octet path: representatives and chunk
// maxima are the top 16 bits of keys, and kappa searches 32-bit keys):
//  1. the lanes stream the row's interior 32-byte chunks (chunk k to lane
//     k mod 32, two loads in flight) and keep, per element position, the raw
//     maximum and minimum: 16 representatives per lane, 512 per row, each
//     the largest key of a distinct set of elements; the row is asked into
//     L2 first, 4 KB per lane;
//  2. theta: for K' <= 32 the K'-th largest of the lanes' largest
//     representatives (a bitonic sort across the warp), else a binary
//     search over the representatives' counts stopped at a 16-key interval:
//     a bound that at least K' representatives, so K' elements, reach;
//  3. the chunks are read again (L2 hits, the next chunk in flight) and the
//     elements >= theta are appended to a 256-entry list in id order, placed
//     by a warp-wide scan; rows of at most 256 non-forced blocks skip steps
//     1-2 and take every element;
//  4. kappa, the K'-th largest candidate, by a binary search over the
//     candidates (8 per lane); those above it are kept, and of those equal
//     to it the first in id order, as many as K' still needs; the kept ids,
//     already in id order, go to the sorted list;
//  5. the row path's outputs (ids, and in fused mode the table).
// A row whose candidates overflow the list is redone by the warp on the row
// path.
// ===========================================================================

// Per lane: how many of the 2 NW packed signed keys are >= t (t > -32768).
template <int NW>
__device__ __forceinline__ int count_ge16(const uint32_t (&w)[NW], int32_t t) {
    const uint32_t t2 = ((uint32_t)(t - 1) & 0xFFFFu) * 0x10001u;
    uint32_t acc = 0;
#pragma unroll
    for (int x = 0; x < NW; ++x) acc += min_u16x2(max_s16x2(w[x], t2) ^ t2, 0x00010001u);
    return (int)((acc & 0xFFFFu) + (acc >> 16));
}

template <int NW>
__device__ __forceinline__ int32_t max16(const uint32_t (&w)[NW]) {
    uint32_t m = w[0];
#pragma unroll
    for (int x = 1; x < NW; ++x) m = max_s16x2(m, w[x]);
    return max((int32_t)(int16_t)(uint16_t)m, (int32_t)(int16_t)(uint16_t)(m >> 16));
}

// LIST: the rows are the long_count entries of long_list (the pair or octet
// path's long rows) and the grid is persistent; else rows 0 .. P.rows - 1.
template <int FM, bool LIST, bool BF16>
__global__ void __launch_bounds__(kWideWarps * 32) wide_select_kernel(const KernelParams P) {
    constexpr int S = BF16 ? 2 : 4;        // element bytes
    constexpr int CE = 32 / S;             // elements per 32-byte chunk
    constexpr int32_t kKeyMin = BF16 ? -32768 : INT32_MIN;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    WideSmem& sm = *reinterpret_cast<WideSmem*>(smem_raw + (size_t)warp * sizeof(WideSmem));
    const SelectArgs& a = P.a;
    const int64_t stride = (int64_t)gridDim.x * kWideWarps;
    const int64_t nrows = LIST ? (int64_t)P.long_count[0] : P.rows;
    // LIST: after its first row (by position) each warp takes the next
    // listed row from a second counter, so that rows of unequal length and
    // late CTAs balance; a list no longer than the grid needs no counter
    auto next_item = [&](int64_t i) -> int64_t {
        if constexpr (LIST) {
            if (nrows <= stride) return nrows;
            uint32_t n = 0;
            if (lane == 0) n = atomicAdd(P.long_count + 1, 1u);
            return stride + (int64_t)__shfl_sync(kFull, n, 0);
        } else {
            return i;
        }
    };

    for (int64_t i = (int64_t)blockIdx.x * kWideWarps + warp; i < nrows;
         i = next_item(i + stride)) {
        const int64_t row = LIST ? (int64_t)P.long_list[i] : i;
        const RowInfo r = row_info_from<FM>(a, row, row_meta<FM>(a, row));
        if (!r.need) {
            write_outputs(P, row, r.t, r.h, r.n, r.lo, r.hi, r.kp, r.all, sm.c.sorted,
                          r.causal_len, r.req, lane);
            __syncwarp();
            continue;
        }

        // ---- geometry of the non-forced range [lo, hi), 32-byte chunks ----
        const char* row_ptr = reinterpret_cast<const char*>(a.scores) +
                              ((int64_t)r.t * a.token_stride + (int64_t)r.h * a.head_stride) * S;
        const uintptr_t a_lo = reinterpret_cast<uintptr_t>(row_ptr) + (uintptr_t)r.lo * S;
        const uintptr_t a_hi = reinterpret_cast<uintptr_t>(row_ptr) + (uintptr_t)r.hi * S;
        const uintptr_t c0 = a_lo & ~(uintptr_t)31;
        const int nchunk = (int)((a_hi - c0 + 31) >> 5);
        const int base_id = r.lo - (int)((a_lo - c0) / S);
        {
            // the whole range towards L2, 4 KB per lane (a row is at most 128 KB)
            uintptr_t plo = c0 < P.buf_lo ? (P.buf_lo + 15) & ~(uintptr_t)15 : c0;
            uintptr_t phi = c0 + ((uintptr_t)nchunk << 5);
            if (phi > P.buf_hi) phi = P.buf_hi & ~(uintptr_t)15;
            const uintptr_t at = plo + ((uintptr_t)lane << 12);
            if (at < phi) prefetch_l2(at, (uint32_t)min((uintptr_t)4096, phi - at));
        }
        const int kp = r.kp;

        // ---- steps 1-2: representatives and theta ----
        int32_t theta = kKeyMin;
        if (r.hi - r.lo > kWideCand) {
            // bf16: a raw maximum and minimum per element position (16 per
            // lane); fp32: the key maximum per position in two sets by the
            // chunk's parity (16 per lane), packed as the top 16 bits below
            uint32_t rmx[8], rmn[8];
            int32_t ra[8], rb[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                rmx[x] = 0x80008000u;
                rmn[x] = 0x7FFF7FFFu;
                ra[x] = rb[x] = INT32_MIN;
            }
            // interior chunks 1 .. nchunk - 2; the edge chunks are left out.
            // Rows of up to kWideHotChunks chunks also keep each chunk's
            // maximum (bf16: raw; fp32: the top 16 bits of its key maximum),
            // so that pass 2 reads only the chunks that reach theta.
            const bool track = nchunk <= kWideHotChunks;
            auto fold = [&](uint32_t (&w)[8], int k, bool second) {
                if constexpr (BF16) {
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        rmx[x] = max_s16x2(rmx[x], w[x]);
                        rmn[x] = min_s16x2(rmn[x], w[x]);
                    }
                    if (track) sm.cmax[k] = (int16_t)max16(w);
                } else {
                    chunk_to_keys<false>(w);
                    int32_t km = INT32_MIN;
#pragma unroll
                    for (int x = 0; x < 8; ++x) {
                        if (second) rb[x] = max(rb[x], (int32_t)w[x]);
                        else ra[x] = max(ra[x], (int32_t)w[x]);
                        km = max(km, (int32_t)w[x]);
                    }
                    if (track) sm.cmax[k] = (int16_t)(km >> 16);
                }
            };
            const int klast = nchunk - 2;
            int k = lane == 0 ? 32 : lane;
            const bool any_interior = k <= klast;
            for (; k + 32 <= klast; k += 64) {
                uint32_t w0[8], w1[8];
                ld32(c0 + ((uintptr_t)k << 5), w0);
                ld32(c0 + ((uintptr_t)(k + 32) << 5), w1);
                fold(w0, k, false);
                fold(w1, k + 32, true);
            }
            if (k <= klast) {
                uint32_t w0[8];
                ld32(c0 + ((uintptr_t)k << 5), w0);
                fold(w0, k, false);
            }
            uint32_t rp[8];   // 16 packed 16-bit representatives
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                if constexpr (BF16) {
                    // a position's largest key: its raw maximum when that is
                    // non-negative, else the key of its raw minimum
                    const uint32_t mneg = sign_mask16(rmx[x]);
                    rp[x] = any_interior ? (rmx[x] & ~mneg) | ((rmn[x] ^ 0x7FFF7FFFu) & mneg)
                                         : 0x80008000u;
                } else {
                    // the top 16 bits of the key maxima (a lower bound of each)
                    const int32_t* src = x < 4 ? ra : rb;
                    const int y = 2 * (x & 3);
                    rp[x] = ((uint32_t)src[y] >> 16) | ((uint32_t)src[y + 1] & 0xFFFF0000u);
                }
            }
            if (kp <= 32) {
                // the kp-th largest of the lanes' largest representatives
                // (a bitonic sort across the warp, descending): kp lanes each
                // hold a representative at or above it
                int32_t v = max16(rp);
#pragma unroll
                for (int kk = 2; kk <= 32; kk <<= 1) {
#pragma unroll
                    for (int jj = kk >> 1; jj > 0; jj >>= 1) {
                        const int32_t o = __shfl_xor_sync(kFull, v, jj);
                        const bool desc = (lane & kk) == 0;
                        const bool lower = (lane & jj) == 0;
                        v = (lower == desc) ? max(v, o) : min(v, o);
                    }
                }
                theta = __shfl_sync(kFull, v, kp - 1);
                if constexpr (!BF16) theta = (int32_t)((uint32_t)theta << 16);
            } else {
                // count(>= lo) >= kp throughout (every representative counts
                // at the smallest key); stop at a 16-key interval
                int32_t lo = kKeyMin, hi = __reduce_max_sync(kFull, max16(rp)) + 1;
                while (hi - lo > 16) {
                    const int32_t mid = (lo + hi) >> 1;
                    if ((int)__reduce_add_sync(kFull, (unsigned)count_ge16(rp, mid)) >= kp) lo = mid;
                    else hi = mid;
                }
                theta = BF16 ? lo : (int32_t)((uint32_t)lo << 16);
            }
        }

        // ---- step 3: candidates >= theta, in id order ----
        const bool raw_ok = theta >= 0;   // raw signed order is key order against it
        // the chunks to read: with theta >= 0 and the chunk maxima kept, the
        // edge chunks and the interior chunks whose raw maximum reaches theta
        // (raw order is key order against a non-negative theta), ascending
        const bool use_hot = raw_ok && r.hi - r.lo > kWideCand && nchunk <= kWideHotChunks;
        int nread = nchunk;
        if (use_hot) {
            int tot = 0;
            for (int b0 = 0; b0 < nchunk; b0 += 32) {
                const int k = b0 + lane;
                const bool hot = k < nchunk && (k == 0 || k == nchunk - 1 ||
                                                (int32_t)sm.cmax[k] >= (BF16 ? theta : theta >> 16));
                const unsigned hb = __ballot_sync(kFull, hot);
                if (hot) sm.hot[tot + __popc(hb & lanemask_lt())] = (uint16_t)k;
                tot += __popc(hb);
            }
            nread = tot;
            __syncwarp();
        }
        auto chunk_at = [&](int i) { return use_hot ? (int)sm.hot[i] : i; };
        const int steps = (nread + 31) >> 5;
        int cbase = 0;
        auto plain = [&](int k) {
            const uintptr_t addr = c0 + ((uintptr_t)k << 5);
            return (k != 0 && k != nchunk - 1) || (addr >= P.buf_lo && addr + 32 <= P.buf_hi);
        };
        uint32_t nx[8];
        auto issue = [&](int st) {
            const int i = lane + 32 * st;
            if (i < nread) {
                const int k = chunk_at(i);
                if (plain(k)) ld32(c0 + ((uintptr_t)k << 5), nx);
            }
        };
        issue(0);
        for (int st = 0; st < steps; ++st) {
            const bool has = lane + 32 * st < nread;
            const int k = has ? chunk_at(lane + 32 * st) : 0;
            uint32_t w[8];
            uint32_t m = 0;
            if (has) {
                if (!plain(k)) {
                    // masked keys, which compare like raw bits against theta >= 0
                    pair_load_edge<BF16>(P, k, c0, base_id, r.lo, r.hi, row_ptr, w);
                } else {
#pragma unroll
                    for (int x = 0; x < 8; ++x) w[x] = nx[x];
                    if (!raw_ok) chunk_to_keys<BF16>(w);
                }
            }
            issue(st + 1);
            if (has) {
                if (theta == kKeyMin) {
                    m = (1u << CE) - 1u;
                } else if constexpr (BF16) {
                    m = ge_bits16<8>(w, theta);
                } else {
#pragma unroll
                    for (int x = 0; x < 8; ++x) m |= ((int32_t)w[x] >= theta ? 1u : 0u) << x;
                }
                if (k == 0 || k == nchunk - 1) {
                    const int first_id = base_id + k * CE;
                    const int lo_e = min(max(r.lo - first_id, 0), CE);
                    const int hi_e = min(max(r.hi - first_id, 0), CE);
                    m &= ((1u << hi_e) - 1u) & ~((1u << lo_e) - 1u);
                }
            }
            int tot;
            const int off = warp_excl_scan(__popc(m), lane, tot);
            if (m) {
                uint32_t* scr = sm.scratch[lane];
#pragma unroll
                for (int x = 0; x < 8; ++x) scr[x] = w[x];
                const int first_id = base_id + k * CE;
                int pos = cbase + off;
                while (m) {
                    const int e = __ffs(m) - 1;
                    m &= m - 1;
                    if (pos < kWideCand) {
                        if constexpr (BF16) sm.c.ckey[pos] = reinterpret_cast<const int16_t*>(scr)[e];
                        else sm.c.ckey32[pos] = (int32_t)scr[e];
                        sm.c.cid[pos] = (uint16_t)(first_id + e);
                    }
                    ++pos;
                }
            }
            cbase += tot;
        }
        __syncwarp();
        if (cbase > kWideCand) {
            // overflow: the whole warp redoes the row on the row path
            warp_item<BF16, 4, 2>(P, row, 0, sm.fallback,
                                  reinterpret_cast<int32_t*>(sm.fallback + P.cap), lane);
            __syncwarp();
            continue;
        }

        // ---- step 4: kappa, the K'-th largest candidate key ----
        // lane holds list positions 8 lane .. 8 lane + 7; padding holds the
        // smallest key, which no searched threshold (> lo >= the smallest
        // key) counts.  count(>= lo) >= K' > count(>= hi) = cnt_hi throughout.
        const int nvalid = min(max(cbase - 8 * lane, 0), 8);
        const uint32_t valid = (1u << nvalid) - 1u;
        uint32_t gtm = 0, eqm = 0;
        int cnt_hi = 0;
        if constexpr (BF16) {
            uint32_t kw[4];
            {
                const uint4 v = *reinterpret_cast<const uint4*>(&sm.c.ckey[8 * lane]);
                kw[0] = v.x; kw[1] = v.y; kw[2] = v.z; kw[3] = v.w;
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    const uint32_t keep = ((valid >> (2 * x)) & 1u ? 0x0000FFFFu : 0u) |
                                          ((valid >> (2 * x + 1)) & 1u ? 0xFFFF0000u : 0u);
                    kw[x] = (kw[x] & keep) | (0x80008000u & ~keep);
                }
            }
            int32_t lo = theta, hi = __reduce_max_sync(kFull, max16(kw)) + 1;
            while (hi - lo > 1) {
                const int32_t mid = (lo + hi) >> 1;
                const int cnt = (int)__reduce_add_sync(kFull, (unsigned)count_ge16(kw, mid));
                if (cnt >= kp) {
                    lo = mid;
                } else {
                    hi = mid;
                    cnt_hi = cnt;
                }
            }
            // kappa = lo: every candidate above it, and the first (K' - count
            // above) of those equal to it, in id order
            gtm = ge_bits16<4>(kw, lo + 1) & valid;
            eqm = (lo == kKeyMin ? valid : ge_bits16<4>(kw, lo) & valid) & ~gtm;
        } else {
            int32_t kk[8];
            {
                const int4* src = reinterpret_cast<const int4*>(&sm.c.ckey32[8 * lane]);
                const int4 u0 = src[0], u1 = src[1];
                kk[0] = u0.x; kk[1] = u0.y; kk[2] = u0.z; kk[3] = u0.w;
                kk[4] = u1.x; kk[5] = u1.y; kk[6] = u1.z; kk[7] = u1.w;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (!((valid >> e) & 1u)) kk[e] = INT32_MIN;
            }
            int32_t mx = kk[0];
#pragma unroll
            for (int e = 1; e < 8; ++e) mx = max(mx, kk[e]);
            int64_t lo = theta, hi = (int64_t)__reduce_max_sync(kFull, mx) + 1;
            while (hi - lo > 1) {
                const int64_t mid = lo + ((hi - lo) >> 1);
                const int32_t t = (int32_t)mid;
                int c = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) c += kk[e] >= t ? 1 : 0;
                const int cnt = (int)__reduce_add_sync(kFull, (unsigned)c);
                if (cnt >= kp) {
                    lo = mid;
                } else {
                    hi = mid;
                    cnt_hi = cnt;
                }
            }
            const int32_t kappa = (int32_t)lo;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const bool vd = (valid >> e) & 1u;
                if (vd && kk[e] > kappa) gtm |= 1u << e;
                if (vd && kk[e] == kappa) eqm |= 1u << e;
            }
        }
        int tall;
        const int tb = warp_excl_scan(__popc(eqm), lane, tall);
        const int allowed = min(max(kp - cnt_hi - tb, 0), __popc(eqm));
        uint32_t rest = eqm;
        for (int i = 0; i < allowed; ++i) rest &= rest - 1;
        uint32_t selm = gtm | (eqm & ~rest);
        int stot;
        int o = warp_excl_scan(__popc(selm), lane, stot);
        while (selm) {
            const int e = __ffs(selm) - 1;
            selm &= selm - 1;
            sm.c.sorted[o++] = sm.c.cid[8 * lane + e];
        }
        __syncwarp();

        // ---- step 5: outputs ----
        write_outputs(P, row, r.t, r.h, r.n, r.lo, r.hi, kp, false, sm.c.sorted, r.causal_len,
                      r.req, lane);
        __syncwarp();
    }
}

template <bool BF16>
cudaError_t launch_wide(const KernelParams& P, const bsa_launch_policy_t& pol, cudaStream_t st) {
    auto kern = P.a.fused ? wide_select_kernel<kFusedYes, false, BF16>
                          : wide_select_kernel<kFusedNo, false, BF16>;
    kern<<<pol.grid, kWideWarps * 32, pol.smem_bytes, st>>>(P);
    return cudaGetLastError();
}

// The second launch of a pair / octet call with long_rows: the listed rows.
cudaError_t launch_wide_list(const KernelParams& P, const bsa_launch_policy_t& pol,
                             cudaStream_t st) {
    if (P.cap > kWideMaxCap || pol.long_grid < 1) return cudaErrorInvalidValue;
    const bool bf16 = P.a.dtype == BSA_DTYPE_BF16;
    auto kern = P.a.fused ? (bf16 ? wide_select_kernel<kFusedYes, true, true>
                                  : wide_select_kernel<kFusedYes, true, false>)
                          : (bf16 ? wide_select_kernel<kFusedNo, true, true>
                                  : wide_select_kernel<kFusedNo, true, false>);
    kern<<<pol.long_grid, kWideWarps * 32, kWideWarps * (int)sizeof(WideSmem), st>>>(P);
    return cudaGetLastError();
}

template <bool BF16, int FM>
cudaError_t launch_pair_fm(const KernelParams& P, const bsa_launch_policy_t& pol,
                           cudaStream_t st) {
    const bool small = P.a.K - P.a.num_init - P.a.num_local <= 16;
    auto kern = small ? pair_select_kernel<BF16, true, FM> : pair_select_kernel<BF16, false, FM>;
    if (pol.smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             pol.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    kern<<<pol.grid, kPairWarps * 32, pol.smem_bytes, st>>>(P);
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_pair(const KernelParams& P, const bsa_launch_policy_t& pol, cudaStream_t st) {
    return P.a.fused ? launch_pair_fm<BF16, kFusedYes>(P, pol, st)
                     : launch_pair_fm<BF16, kFusedNo>(P, pol, st);
}

template <bool BF16, int R>
cudaError_t launch_group_t(const KernelParams& P, const bsa_launch_policy_t& pol,
                           cudaStream_t st) {
    // K' <= K - num_init - num_local: a 16-entry id sort suffices for K' <= 16
    const bool small = P.a.K - P.a.num_init - P.a.num_local <= 16;
    auto kern = small ? group_select_kernel<BF16, R, true> : group_select_kernel<BF16, R, false>;
    if (pol.smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             pol.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    kern<<<pol.grid, kThreads, pol.smem_bytes, st>>>(P);
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_group(const KernelParams& P, const bsa_launch_policy_t& pol,
                         cudaStream_t st) {
    return launch_group_t<BF16, 8>(P, pol, st);
}

template <bool BF16, int NV, int R>
cudaError_t launch_t(const KernelParams& P, const bsa_launch_policy_t& pol, cudaStream_t st) {
    auto kern = select_kernel<BF16, NV, R>;
    if (pol.smem_bytes > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             pol.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    kern<<<pol.grid, kThreads, pol.smem_bytes, st>>>(P);
    return cudaGetLastError();
}

template <bool BF16, int NV>
cudaError_t launch_nv(const KernelParams& P, const bsa_launch_policy_t& pol, cudaStream_t st) {
    switch (pol.reps_per_lane) {
        case 1: return launch_t<BF16, NV, 1>(P, pol, st);
        case 2: return launch_t<BF16, NV, 2>(P, pol, st);
        default: return launch_t<BF16, NV, 2 * NV>(P, pol, st);
    }
}

template <bool BF16>
cudaError_t launch_dt(const KernelParams& P, const bsa_launch_policy_t& pol, cudaStream_t st) {
    switch (pol.vecs_per_lane) {
        case 1: return launch_nv<BF16, 1>(P, pol, st);
        case 2: return launch_nv<BF16, 2>(P, pol, st);
        default: return launch_nv<BF16, 4>(P, pol, st);
    }
}

// ===========================================================================
// Fused index score + select for decode rows.
//
// The decode side of the indexer first writes block scores into the unified
// buffer and then selects from it (vLLM PR #47502 report, 实现拆解 items
// 1-3: minimax_m3_index_decode_score with score_out = unified_scores[:nd],
// then one top-k pass).  The pages do not print the score formula; the
// reading taken is one pooled index key per physical 128-token block (page =
// sparse block = index-K block, section 关键源码片段), shared by the index
// heads, with
//     score[t, h, b] = sum over d of q[t, h, d] * k[block_table[req, b], d]
// accumulated in fp32 and no scale factor (item 6 removed sm_scale).
//
// A CTA of 4 warps takes one group of R requests, R = max(1, 4 / (dql * H)),
// so that each warp has about one row to select; the grid has one CTA per
// group and the hardware balances CTAs of unequal length (requests differ in
// their causal block counts).  The group's query rows are staged in shared
// memory as fp32 and the causal blocks are scored in one of two ways:
//  * segment scoring (D = 64 or 128 and at most 4 query rows per request):
//    a segment of D / 8 lanes reads one key row with one 16-byte load per
//    lane, so that a warp-wide load covers whole rows (two of D = 128, four
//    of D = 64) and a warp keeps 32 rows in flight.  Each lane holds its 8
//    dimensions of every query row in registers and forms 8-term partial dot
//    products for the segment's D / 8 rows; a reduce-scatter over the
//    segment's lanes (recursive halving with shuffles) leaves each lane with
//    the full dot products of one row.  The warps of the CTA take 32-block
//    rounds of the group's requests in turn, each loading its next round's
//    table entries one round ahead.
//  * thread scoring (every other D and query count): a thread takes one
//    causal block at a time, reads its key row as 16-byte vectors and scores
//    it against every query row of the request.
// The scores of the causal blocks go into the caller's unified buffer, and
// after a block barrier the CTA's warps select the top-k of the group's rows
// from that buffer with the warp path, reading through L2 what the CTA has
// just written (no second launch and no re-read from HBM).  A causal block
// whose table entry is missing (b >= max_blocks) or out of range scores -inf.
// ===========================================================================
constexpr int kScoreThreads = 128;
constexpr int kScoreWarps = kScoreThreads / 32;
constexpr int kScoreRows = 4;        // query rows per group when dql * H is small
constexpr int kSegMaxQ = 4;          // segment scoring takes up to 4 query rows per request

struct ScoreParams {
    KernelParams P;          // the selection over the score buffer (fp32, decode rows)
    const uint16_t* q;       // bf16 [T, H, D]
    const uint16_t* k;       // bf16 [nb, D]
    int64_t nb;
    int32_t D;
    int32_t nq;              // dql * H query rows per request
    int32_t group;           // requests a CTA takes at a time
    float* scores;           // element (t, h, b) at t * token_stride + h * head_stride + b
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ int64_t causal_blocks_of(int64_t len, int64_t M) {
    int64_t v = len > 0 ? (len + kPageSize - 1) >> kLogPageSize : 0;
    return v < M ? v : M;
}

// Writes block b's score for query row x of request req if b is below that
// row's causal count.
__device__ __forceinline__ void store_score(const ScoreParams& S, int64_t req, int64_t seq, int x,
                                            int64_t b, float val) {
    const SelectArgs& a = S.P.a;
    const int lq = x / (int)a.H;
    const int h = x - lq * (int)a.H;
    if (b < causal_blocks_of(seq - a.dql + lq + 1, a.M)) {
        const int64_t t = req * a.dql + lq;
        S.scores[t * a.token_stride + h * a.head_stride + b] = val;
    }
}

__device__ __forceinline__ float dot8(const float (&kf)[8], const float (&qv)[8], float acc) {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(kf[e], qv[e], acc);
    return acc;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& kv, float (&kf)[8]) {
    kf[0] = bf16_lo(kv.x); kf[1] = bf16_hi(kv.x); kf[2] = bf16_lo(kv.y); kf[3] = bf16_hi(kv.y);
    kf[4] = bf16_lo(kv.z); kf[5] = bf16_hi(kv.z); kf[6] = bf16_lo(kv.w); kf[7] = bf16_hi(kv.w);
}

// Thread scoring of the group's requests (any D that is a multiple of 8).
template <int NQ>
__device__ __forceinline__ void score_group_threads(const ScoreParams& S, int64_t req0, int nreq,
                                                    const float* qs, int tid) {
    const SelectArgs& a = S.P.a;
    const int D = S.D;
    const int nq = S.nq;
    for (int rr = 0; rr < nreq; ++rr) {
        const int64_t req = req0 + rr;
        const float* qr = qs + (size_t)rr * nq * D;
        const int64_t seq = __ldg(a.seq_lens + req);
        // the last query row (local_q = dql - 1, position seq - 1) has the
        // most causal blocks
        const int64_t vmax = causal_blocks_of(seq, a.M);
        const int32_t* table = a.block_table + req * a.max_blocks;
        for (int64_t b = tid; b < vmax; b += kScoreThreads) {
            float acc[NQ];
#pragma unroll
            for (int x = 0; x < NQ; ++x) acc[x] = 0.f;
            const int64_t phys = b < a.max_blocks ? (int64_t)__ldg(table + b) : -1;
            const bool ok = phys >= 0 && phys < S.nb;
            report_status(a.status, b < a.max_blocks && !ok, BSA_STATUS_BAD_BLOCK_ID);
            if (ok) {
                const uint4* kr = reinterpret_cast<const uint4*>(S.k + phys * D);
#pragma unroll 8
                for (int c = 0; c < D / 8; ++c) {
                    float kf[8];
                    unpack_bf16x8(__ldg(kr + c), kf);
#pragma unroll
                    for (int x = 0; x < NQ; ++x) {
                        if (x < nq) {
                            const float4* qv = reinterpret_cast<const float4*>(qr + x * D + 8 * c);
                            const float4 q0 = qv[0], q1 = qv[1];
                            const float qf[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                            acc[x] = dot8(kf, qf, acc[x]);
                        }
                    }
                }
            }
#pragma unroll
            for (int x = 0; x < NQ; ++x)
                if (x < nq) store_score(S, req, seq, x, b, ok ? acc[x] : __int_as_float(0xFF800000));
        }
    }
}

// Segment scoring of the group's requests: SL = D / 8 lanes per key row.
template <int NQ, int SL>
__device__ __forceinline__ void score_group_segments(const ScoreParams& S, int64_t req0, int nreq,
                                                     const float* qs, int warp, int lane) {
    constexpr int SEGS = 32 / SL;     // key rows per warp-wide load
    constexpr int D = 8 * SL;
    const SelectArgs& a = S.P.a;
    const int nq = S.nq;
    const int sg = lane / SL;         // this lane's segment
    const int j = lane % SL;          // its 8 dimensions [8 j, 8 j + 8)
    // 32-block rounds over the group's requests, flattened: the warp takes
    // rounds warp, warp + 4, ...; `before` counts the rounds of earlier requests
    int64_t next = warp, before = 0;
    for (int rr = 0; rr < nreq; ++rr) {
        const int64_t req = req0 + rr;
        const int64_t seq = __ldg(a.seq_lens + req);
        const int64_t vmax = causal_blocks_of(seq, a.M);
        const int64_t rounds = (vmax + 31) >> 5;
        if (next < before + rounds) {
            const int32_t* table = a.block_table + req * a.max_blocks;
            const int64_t tab_end = vmax < a.max_blocks ? vmax : a.max_blocks;
            float qv[NQ][8];
            const float* qr = qs + (size_t)rr * nq * D + 8 * j;
#pragma unroll
            for (int x = 0; x < NQ; ++x) {
                float4 q0 = make_float4(0.f, 0.f, 0.f, 0.f), q1 = q0;
                if (x < nq) {
                    q0 = *reinterpret_cast<const float4*>(qr + x * D);
                    q1 = *reinterpret_cast<const float4*>(qr + x * D + 4);
                }
                qv[x][0] = q0.x; qv[x][1] = q0.y; qv[x][2] = q0.z; qv[x][3] = q0.w;
                qv[x][4] = q1.x; qv[x][5] = q1.y; qv[x][6] = q1.z; qv[x][7] = q1.w;
            }
            // each lane keeps the table entry of its block in the warp's next
            // round, loaded one round ahead
            int32_t tbn;
            {
                const int64_t base = (next - before) << 5;
                tbn = base + lane < tab_end ? __ldg(table + base + lane) : -1;
            }
            for (; next < before + rounds; next += kScoreWarps) {
                const int64_t base = (next - before) << 5;
                // lane l holds the table entry of block base + l (-1 past the table)
                const int32_t tb = tbn;
                {
                    const int64_t nb2 = base + 32 * kScoreWarps + lane;
                    tbn = nb2 < tab_end ? __ldg(table + nb2) : -1;
                }
                uint4 kv[SL];
#pragma unroll
                for (int i = 0; i < SL; ++i) {   // row i of the segment: block base + sg + SEGS i
                    const int64_t phys = __shfl_sync(kFull, tb, sg + SEGS * i);
                    kv[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (phys >= 0 && phys < S.nb)
                        kv[i] = __ldg(reinterpret_cast<const uint4*>(S.k + phys * D) + j);
                }
                float acc[SL][NQ];
#pragma unroll
                for (int i = 0; i < SL; ++i) {
                    float kf[8];
                    unpack_bf16x8(kv[i], kf);
#pragma unroll
                    for (int x = 0; x < NQ; ++x) acc[i][x] = dot8(kf, qv[x], 0.f);
                }
                // reduce-scatter over the segment: at distance m the lanes with
                // bit m set keep the upper half of the rows and the others the
                // lower half, each adding its partner's partial sums of the
                // half it keeps; lane j ends with row j
#pragma unroll
                for (int m = SL / 2; m >= 1; m >>= 1) {
                    const bool up = (j & m) != 0;
#pragma unroll
                    for (int i = 0; i < m; ++i) {
#pragma unroll
                        for (int x = 0; x < NQ; ++x) {
                            const float keep = up ? acc[i + m][x] : acc[i][x];
                            const float send = up ? acc[i][x] : acc[i + m][x];
                            acc[i][x] = keep + __shfl_xor_sync(kFull, send, m);
                        }
                    }
                }
                const int own = sg + SEGS * j;           // this lane's block, relative to base
                const int64_t ph = __shfl_sync(kFull, tb, own);
                const bool ok = ph >= 0 && ph < S.nb;
                report_status(a.status, base + own < tab_end && !ok, BSA_STATUS_BAD_BLOCK_ID);
#pragma unroll
                for (int x = 0; x < NQ; ++x)
                    if (x < nq)
                        store_score(S, req, seq, x, base + own,
                                    ok ? acc[0][x] : __int_as_float(0xFF800000));
            }
        }
        before += rounds;
    }
}

// SL = 0: thread scoring; SL = 8 or 16: segment scoring with D = 8 SL.
template <int NQ, int SL>
__global__ void __launch_bounds__(kScoreThreads, 4) index_score_select_kernel(const ScoreParams S) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int D = S.D;
    const int nq = S.nq;
    const int R = S.group;
    const SelectArgs& a = S.P.a;
    float* qs = reinterpret_cast<float*>(smem_raw);                       // [R * nq][D]
    const size_t qbytes = ((size_t)R * nq * D * 4 + 15) & ~(size_t)15;
    uint32_t* s_keys = reinterpret_cast<uint32_t*>(smem_raw + qbytes) + (size_t)warp * S.P.cap * 2;
    int32_t* s_ids = reinterpret_cast<int32_t*>(s_keys + S.P.cap);
    const int64_t B = a.T / a.dql;
    const int64_t ngroups = (B + R - 1) / R;
    for (int64_t grp = blockIdx.x; grp < ngroups; grp += gridDim.x) {
        const int64_t req0 = grp * R;
        const int nreq = (int)min((int64_t)R, B - req0);
        __syncthreads();   // the previous group's readers of qs are done
        // the group's query rows are contiguous: rows (req0 * dql + lq) * H + h
        const uint16_t* qsrc = S.q + req0 * (int64_t)nq * D;
        for (int i = tid; i < nreq * nq * D; i += kScoreThreads)
            qs[i] = __uint_as_float((uint32_t)qsrc[i] << 16);
        __syncthreads();
        if constexpr (SL == 0)
            score_group_threads<NQ>(S, req0, nreq, qs, tid);
        else
            score_group_segments<NQ, SL>(S, req0, nreq, qs, warp, lane);
        __syncthreads();   // the group's scores are visible to the whole CTA
        for (int x = warp; x < nreq * nq; x += kScoreWarps) {
            warp_item<false, 4, 2, true>(S.P, req0 * nq + x, 0, s_keys, s_ids, lane);
            __syncwarp();
        }
    }
}

template <int NQ, int SL>
cudaError_t launch_score(const ScoreParams& S, int grid, size_t smem, cudaStream_t st) {
    auto kern = index_score_select_kernel<NQ, SL>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<grid, kScoreThreads, smem, st>>>(S);
    return cudaGetLastError();
}

template <int SL>
cudaError_t launch_score_seg(const ScoreParams& S, int grid, size_t smem, cudaStream_t st) {
    if (S.nq <= 1) return launch_score<1, SL>(S, grid, smem, st);
    if (S.nq <= 2) return launch_score<2, SL>(S, grid, smem, st);
    return launch_score<4, SL>(S, grid, smem, st);
}

}  // namespace

cudaError_t launch_select(const SelectArgs& a, const bsa_launch_policy_t& pol,
                          const SplitWorkspace& ws, cudaStream_t stream) {
    KernelParams P;
    P.a = a;
    P.a.status = current_status_word();
    div_magic((uint32_t)(a.H > 0 ? a.H : 1), &P.a.h_mul, &P.a.h_shift);
    div_magic((uint32_t)(a.dql > 0 ? a.dql : 1), &P.a.dql_mul, &P.a.dql_shift);
    P.ws = Split{ws.keys, ws.ids, ws.counts, ws.tickets};
    P.long_list = nullptr;
    P.long_count = nullptr;
    P.chunks_per_row = pol.chunks_per_row;
    P.cap = pol.cand_capacity;
    P.rows = a.T * a.H;
    const int vec = a.dtype == BSA_DTYPE_BF16 ? 8 : 4;
    const int64_t esz = a.dtype == BSA_DTYPE_BF16 ? 2 : 4;
    P.buf_lo = reinterpret_cast<uintptr_t>(a.scores);
    P.buf_hi = P.buf_lo + (uintptr_t)(((a.T > 0 ? a.T - 1 : 0) * a.token_stride +
                                        (a.H > 0 ? a.H - 1 : 0) * a.head_stride + a.M) * esz);
    const int64_t max_vecs = (a.M + vec - 1) / vec + 1;
    int64_t vpc = (max_vecs + pol.chunks_per_row - 1) / pol.chunks_per_row;
    const int64_t pass = 32LL * pol.vecs_per_lane;
    vpc = (vpc + pass - 1) / pass * pass;
    P.vecs_per_chunk = (int32_t)vpc;
    if (P.rows == 0) return cudaSuccess;
    if (pol.path == BSA_PATH_GROUP)
        return a.dtype == BSA_DTYPE_BF16 ? launch_group<true>(P, pol, stream)
                                         : launch_group<false>(P, pol, stream);
    if (pol.long_rows) {
        // rows over 2 KB: listed by the pair / octet kernel, then the wide path
        if (ws.long_list == nullptr || ws.long_count == nullptr ||
            (pol.path != BSA_PATH_PAIR && pol.path != BSA_PATH_OCTET))
            return cudaErrorInvalidValue;
        P.long_list = ws.long_list;
        P.long_count = ws.long_count;
        const bool bf16 = a.dtype == BSA_DTYPE_BF16;
        const cudaError_t e =
            pol.path == BSA_PATH_PAIR
                ? (bf16 ? launch_pair<true>(P, pol, stream) : launch_pair<false>(P, pol, stream))
                : (bf16 ? launch_octet<true>(P, pol, stream) : launch_octet<false>(P, pol, stream));
        if (e != cudaSuccess) return e;
        return launch_wide_list(P, pol, stream);
    }
    if (pol.path == BSA_PATH_PAIR)
        return a.dtype == BSA_DTYPE_BF16 ? launch_pair<true>(P, pol, stream)
                                         : launch_pair<false>(P, pol, stream);
    if (pol.path == BSA_PATH_OCTET)
        return a.dtype == BSA_DTYPE_BF16 ? launch_octet<true>(P, pol, stream)
                                         : launch_octet<false>(P, pol, stream);
    if (pol.path == BSA_PATH_WIDE) {
        if (pol.cand_capacity > kWideMaxCap) return cudaErrorInvalidValue;
        return a.dtype == BSA_DTYPE_BF16 ? launch_wide<true>(P, pol, stream)
                                         : launch_wide<false>(P, pol, stream);
    }
    return a.dtype == BSA_DTYPE_BF16 ? launch_dt<true>(P, pol, stream)
                                     : launch_dt<false>(P, pol, stream);
}

cudaError_t launch_index_score_select(const SelectArgs& a, const uint16_t* q, const uint16_t* k,
                                      int64_t nb, int32_t D, float* scores, cudaStream_t stream) {
    ScoreParams S;
    KernelParams& P = S.P;
    P.a = a;
    P.a.status = current_status_word();
    div_magic((uint32_t)(a.H > 0 ? a.H : 1), &P.a.h_mul, &P.a.h_shift);
    div_magic((uint32_t)(a.dql > 0 ? a.dql : 1), &P.a.dql_mul, &P.a.dql_shift);
    P.ws = Split{nullptr, nullptr, nullptr, nullptr};
    P.long_list = nullptr;
    P.long_count = nullptr;
    P.chunks_per_row = 1;
    // the warp path with 4 fp32 vectors per lane per pass
    P.cap = (a.K + 32 * 4 + 31) / 32 * 32;
    P.rows = a.T * a.H;
    P.buf_lo = reinterpret_cast<uintptr_t>(scores);
    P.buf_hi = P.buf_lo + (uintptr_t)(((a.T > 0 ? a.T - 1 : 0) * a.token_stride +
                                        (a.H > 0 ? a.H - 1 : 0) * a.head_stride + a.M) * 4);
    const int64_t max_vecs = (a.M + 3) / 4 + 1;
    P.vecs_per_chunk = (int32_t)((max_vecs + 127) / 128 * 128);
    S.q = q;
    S.k = k;
    S.nb = nb;
    S.D = D;
    S.nq = (int32_t)(a.dql * a.H);
    S.group = S.nq >= kScoreRows ? 1 : kScoreRows / S.nq;
    S.scores = scores;
    const int64_t B = a.T / a.dql;
    if (B == 0) return cudaSuccess;
    const size_t smem = (((size_t)S.group * S.nq * D * 4 + 15) & ~(size_t)15) +
                        (size_t)kScoreWarps * P.cap * 8;
    const int64_t ngroups = (B + S.group - 1) / S.group;
    int64_t grid = ngroups < INT32_MAX ? ngroups : INT32_MAX;
    if (S.nq <= kSegMaxQ && D == 128) return launch_score_seg<16>(S, (int)grid, smem, stream);
    if (S.nq <= kSegMaxQ && D == 64) return launch_score_seg<8>(S, (int)grid, smem, stream);
    if (S.nq <= 1) return launch_score<1, 0>(S, (int)grid, smem, stream);
    if (S.nq <= 2) return launch_score<2, 0>(S, (int)grid, smem, stream);
    if (S.nq <= 4) return launch_score<4, 0>(S, (int)grid, smem, stream);
    if (S.nq <= 8) return launch_score<8, 0>(S, (int)grid, smem, stream);
    return launch_score<16, 0>(S, (int)grid, smem, stream);
}

}  // namespace bsa
