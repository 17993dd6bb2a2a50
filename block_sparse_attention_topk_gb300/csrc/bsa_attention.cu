// bsa_attention.cu -- sparse decode attention over the page-16 sparse block
// table: the consumer of the selector's table.
//
// What it computes (vLLM PR #47984 report, "[ROCm][MiniMax-M3][Spec Decode]
// Support speculative decode with AITER sparse PA", sections 实现拆解 items
// 1-2: the decode sparse paged attention reads the page-16 table and its
// sparse context length; vLLM PR #47502 report, 实现拆解 item 5: the sparse
// decode kernels take their valid blocks from the sequence position).  The
// pages show only the interface; the readings taken are: index head h
// selects for KV head h, shared by G query heads; the KV cache is paged in
// 16-token pages, bf16 [num_pages, 16, H, D], and a table entry is a page
// id (physical 128-token block * 8 + page); row (t, h) attends to its first
// ctx = sparse_ctx[t, h] tokens in table order, token j in page
// sparse_bt[t, h, j / 16] at slot j % 16; and query head g takes
//     out[t, h, g] = sum_j softmax_j(scale * q[t, h, g] . k_j) v_j.
// A row with an empty context yields zeros, and a token whose page id lies
// outside [0, num_pages) takes no part.
//
// How: one CTA of 8 warps per row (t, h) and all its G query heads; the
// warps split the row's context.  The row's queries sit in shared memory as
// fp32.  Each warp walks its share 32 tokens (two pages) at a time: each
// lane scores one token against every query head (reading the token's key
// row as 16-byte vectors), the warp folds the tile into a running maximum
// and sum per head (online softmax, Milakov and Gimelshein, "Online
// normalizer calculation for softmax", 2018), and then the lanes accumulate
// the tile's value rows weighted by the broadcast probabilities: each lane
// owns 4 (D = 64, 128) or D / 32 dimensions of one token of a warp-wide
// load, so that a load covers two tokens' rows at D = 64 (8 bytes per lane)
// and one row above; the tile's two page ids are read once.  The
// warps' partial maxima, sums and outputs then merge in shared memory (each
// rescaled by exp(its maximum - the overall maximum)).  Decode attention
// moves each key and value once and does O(G) flops per element, so it is
// bound by memory and runs on the CUDA cores.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <climits>

#include "bsa_internal.h"

namespace bsa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kAttnWarps = 8;   // warps sharing one row's context

struct AttnParams {
    const uint16_t* q;       // bf16 [rows, G, D]
    const uint16_t* k;       // bf16 [num_pages, 16, H, D]
    const uint16_t* v;       // bf16 [num_pages, 16, H, D]
    int64_t num_pages;
    const int32_t* bt;       // int32 [rows, width]
    const int32_t* ctx;      // int32 [rows]
    int64_t rows;            // T * H
    int32_t H, G, width;     // width = topk * 8 table entries per row
    float scale;
    float* out;              // fp32 [rows, G, D]
    uint32_t* status;        // the device status word, or null
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, d));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) x += __shfl_xor_sync(kFull, x, d);
    return x;
}

// DL bf16 values at p (DL * 2 bytes, aligned to that) as fp32.
template <int DL>
__device__ __forceinline__ void load_dl(const uint16_t* p, float (&f)[DL]) {
    if constexpr (DL == 2) {
        const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(p));
        f[0] = bf_lo(w);
        f[1] = bf_hi(w);
    } else if constexpr (DL == 4) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
        f[0] = bf_lo(w.x);
        f[1] = bf_hi(w.x);
        f[2] = bf_lo(w.y);
        f[3] = bf_hi(w.y);
    } else {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = bf_lo(ws[i]);
            f[2 * i + 1] = bf_hi(ws[i]);
        }
    }
}

// GP >= G query heads (a power of two), DL = D / 32 dimensions per lane.
// Shared memory: queries [GP][D], then per warp its partial maxima [GP],
// sums [GP] and outputs [GP][D].
// Resident CTAs per SM the register bound asks for: 4 where the lane's
// accumulators are small (a decode batch is often a single wave of CTAs, so
// occupancy decides), 2 for 8 query heads of wide dimensions.
constexpr int attn_ctas(int gp, int dl) { return gp * (dl < 4 ? 4 : dl) <= 16 ? 4 : 2; }

template <int GP, int DL>
__global__ void __launch_bounds__(kAttnWarps * 32, attn_ctas(GP, DL))
sparse_decode_attention_kernel(const AttnParams A) {
    constexpr int D = 32 * DL;
    // value phase: each lane owns VD dimensions of one token of a load; a
    // load covers TPL tokens (D = 64: two tokens, 8 bytes per lane)
    constexpr int VD = DL < 4 ? 4 : DL;
    constexpr int LPT = D / VD;            // lanes per token
    constexpr int TPL = 32 / LPT;          // tokens per warp-wide load
    constexpr int VB = VD >= 8 ? 2 : 4;    // value loads in flight per lane
    extern __shared__ __align__(16) float smem[];
    float* qs = smem;
    float* pm = qs + GP * D;
    float* pl = pm + kAttnWarps * GP;
    float* pacc = pl + kAttnWarps * GP;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int sub = lane / LPT;            // the lane's token within a load
    const int d0 = (lane % LPT) * VD;      // its first value dimension
    const int G = A.G;
    const int cap = A.width * BSA_SUB_PAGE_SIZE;
    const int64_t slot_stride = (int64_t)A.H * D;   // elements between slots of a page
    for (int64_t row = blockIdx.x; row < A.rows; row += gridDim.x) {
        const int h = (int)(row % A.H);
        const int32_t* bt = A.bt + row * A.width;
        const int ctx_in = __ldg(A.ctx + row);
        const int ctx = max(0, min(ctx_in, cap));
        if (threadIdx.x == 0) report_status(A.status, ctx != ctx_in, BSA_STATUS_BAD_CONTEXT);
        const uint16_t* qrow = A.q + row * (int64_t)G * D;
        __syncthreads();   // the previous row's readers of shared memory are done
        for (int i = threadIdx.x; i < G * D; i += kAttnWarps * 32)
            qs[i] = __uint_as_float((uint32_t)__ldg(qrow + i) << 16);
        __syncthreads();
        float m[GP], l[GP], acc[GP][VD];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int d = 0; d < VD; ++d) acc[g][d] = 0.f;
        }
        for (int tile = 32 * warp; tile < ctx; tile += 32 * kAttnWarps) {
            // the tile's two pages (tokens tile .. tile + 15 and tile + 16 .. tile + 31)
            const int32_t pa = __ldg(bt + (tile >> 4));
            const int32_t pb = tile + 16 < ctx ? __ldg(bt + (tile >> 4) + 1) : -1;
            const bool oka = pa >= 0 && pa < A.num_pages;
            const bool okb = pb >= 0 && pb < A.num_pages;
            // the tile's value pages towards L2 while the scores are formed
            if (lane < 2 && (lane == 0 ? oka : okb)) {
                const int64_t pg = lane == 0 ? pa : pb;
                const uint16_t* vp = A.v + pg * BSA_SUB_PAGE_SIZE * slot_stride;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vp),
                             "r"((uint32_t)(BSA_SUB_PAGE_SIZE * slot_stride * 2)) : "memory");
            }
            report_status(A.status, lane == 0 && (!oka || (tile + 16 < ctx && !okb)),
                          BSA_STATUS_BAD_PAGE);
            // ---- scores: lane j of the tile takes token tile + j ----
            const int j = tile + lane;
            const int32_t page = lane < 16 ? pa : pb;
            const bool ok = j < ctx && (lane < 16 ? oka : okb);
            float s[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) s[g] = 0.f;
            if (ok) {
                const uint4* kr = reinterpret_cast<const uint4*>(
                    A.k + ((int64_t)page * BSA_SUB_PAGE_SIZE + (lane & 15)) * slot_stride + (int64_t)h * D);
#pragma unroll 8
                for (int c = 0; c < D / 8; ++c) {
                    const uint4 kv = __ldg(kr + c);
                    const float kf[8] = {bf_lo(kv.x), bf_hi(kv.x), bf_lo(kv.y), bf_hi(kv.y),
                                         bf_lo(kv.z), bf_hi(kv.z), bf_lo(kv.w), bf_hi(kv.w)};
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        if (g < G) {
                            const float4* qv = reinterpret_cast<const float4*>(qs + g * D + 8 * c);
                            const float4 q0 = qv[0], q1 = qv[1];
                            float a = s[g];
                            a = fmaf(kf[0], q0.x, a);
                            a = fmaf(kf[1], q0.y, a);
                            a = fmaf(kf[2], q0.z, a);
                            a = fmaf(kf[3], q0.w, a);
                            a = fmaf(kf[4], q1.x, a);
                            a = fmaf(kf[5], q1.y, a);
                            a = fmaf(kf[6], q1.z, a);
                            a = fmaf(kf[7], q1.w, a);
                            s[g] = a;
                        }
                    }
                }
            }
            // ---- online softmax: fold the tile into the running max / sum ----
            float p[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                const float sg = ok ? s[g] * A.scale : -INFINITY;
                const float mn = fmaxf(m[g], warp_max(sg));
                // mn stays -inf until a usable token has been seen
                const float corr = mn == -INFINITY ? 1.f : expf(m[g] - mn);
                p[g] = ok ? expf(sg - mn) : 0.f;
                l[g] = l[g] * corr + warp_sum(p[g]);
#pragma unroll
                for (int d = 0; d < VD; ++d) acc[g][d] *= corr;
                m[g] = mn;
            }
            // ---- values: lane (sub, d0) takes tokens sub, sub + TPL, ... of
            // the tile, dimensions [d0, d0 + VD); VB rows are loaded before
            // any of them is used ----
            const uint16_t* va = A.v + (int64_t)pa * BSA_SUB_PAGE_SIZE * slot_stride + (int64_t)h * D + d0;
            const uint16_t* vb = A.v + (int64_t)pb * BSA_SUB_PAGE_SIZE * slot_stride + (int64_t)h * D + d0;
#pragma unroll
            for (int i0 = 0; i0 < 32 / TPL; i0 += VB) {
                float vf[VB][VD];
#pragma unroll
                for (int v = 0; v < VB; ++v) {
                    const int u = sub + TPL * (i0 + v);
                    const bool use = tile + u < ctx && (u < 16 ? oka : okb);
                    if (use) {
                        load_dl<VD>((u < 16 ? va : vb) + (int64_t)(u & 15) * slot_stride, vf[v]);
                    } else {
#pragma unroll
                        for (int d = 0; d < VD; ++d) vf[v][d] = 0.f;
                    }
                }
                // tokens past the context or on unusable pages have p = 0
#pragma unroll
                for (int v = 0; v < VB; ++v) {
                    const int u = sub + TPL * (i0 + v);
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        const float pj = __shfl_sync(kFull, p[g], u);
#pragma unroll
                        for (int d = 0; d < VD; ++d) acc[g][d] = fmaf(pj, vf[v][d], acc[g][d]);
                    }
                }
            }
        }
        // the lanes that share dimensions (one per token of a load) add up
#pragma unroll
        for (int t = LPT; t < 32; t <<= 1) {
#pragma unroll
            for (int g = 0; g < GP; ++g)
#pragma unroll
                for (int d = 0; d < VD; ++d) acc[g][d] += __shfl_xor_sync(kFull, acc[g][d], t);
        }
        // ---- merge the warps' partial results ----
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            if (lane == 0) {
                pm[warp * GP + g] = m[g];
                pl[warp * GP + g] = l[g];
            }
            if (sub == 0) {
#pragma unroll
                for (int d = 0; d < VD; ++d) pacc[(warp * GP + g) * D + d0 + d] = acc[g][d];
            }
        }
        __syncthreads();
        float* orow = A.out + row * (int64_t)G * D;
        for (int i = threadIdx.x; i < G * D; i += kAttnWarps * 32) {
            const int g = i / D;
            const int d = i - g * D;
            float mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < kAttnWarps; ++w) mx = fmaxf(mx, pm[w * GP + g]);
            float den = 0.f, num = 0.f;
            if (mx != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kAttnWarps; ++w) {
                    const float mw = pm[w * GP + g];
                    const float e = mw == -INFINITY ? 0.f : expf(mw - mx);
                    den = fmaf(pl[w * GP + g], e, den);
                    num = fmaf(pacc[(w * GP + g) * D + d], e, num);
                }
            }
            orow[i] = den > 0.f ? num / den : 0.f;
        }
    }
}

template <int GP, int DL>
cudaError_t launch_attn(const AttnParams& A, cudaStream_t st) {
    const size_t D = 32 * DL;
    const size_t smem = (GP * D + 2 * kAttnWarps * GP + (size_t)kAttnWarps * GP * D) * sizeof(float);
    auto kern = sparse_decode_attention_kernel<GP, DL>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    // one row per CTA, not capped at the resident CTAs
    int64_t grid = A.rows;
    if (grid > INT32_MAX) grid = INT32_MAX;
    kern<<<(int)grid, kAttnWarps * 32, smem, st>>>(A);
    return cudaGetLastError();
}

template <int DL>
cudaError_t launch_attn_g(const AttnParams& A, cudaStream_t st) {
    if (A.G <= 1) return launch_attn<1, DL>(A, st);
    if (A.G <= 2) return launch_attn<2, DL>(A, st);
    if (A.G <= 4) return launch_attn<4, DL>(A, st);
    return launch_attn<8, DL>(A, st);
}

}  // namespace
}  // namespace bsa

using namespace bsa;

extern "C" int bsa_sparse_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                           int64_t num_pages, const int32_t* sparse_bt,
                                           const int32_t* sparse_ctx, int64_t T, int64_t H,
                                           int64_t G, int64_t D, int32_t K, float scale,
                                           float* out, void* stream) {
    if (T < 0 || H < 1 || num_pages < 0) return BSA_ERR_SHAPE;
    if (G < 1 || G > BSA_MAX_ATTN_GROUP) return BSA_ERR_SHAPE;
    if (D != 64 && D != 128 && D != 256) return BSA_ERR_SHAPE;
    if (K < 1 || K > BSA_MAX_TOPK) return BSA_ERR_TOPK;
    if (T == 0) return BSA_OK;
    if (q == nullptr || sparse_bt == nullptr || sparse_ctx == nullptr || out == nullptr ||
        (num_pages > 0 && (k_cache == nullptr || v_cache == nullptr)))
        return BSA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(q) & 15) != 0 || (reinterpret_cast<uintptr_t>(k_cache) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(v_cache) & 15) != 0 || (reinterpret_cast<uintptr_t>(out) & 3) != 0)
        return BSA_ERR_ALIGN;
    AttnParams A;
    A.q = static_cast<const uint16_t*>(q);
    A.k = static_cast<const uint16_t*>(k_cache);
    A.v = static_cast<const uint16_t*>(v_cache);
    A.num_pages = num_pages;
    A.bt = sparse_bt;
    A.ctx = sparse_ctx;
    A.rows = T * H;
    A.H = (int32_t)H;
    A.G = (int32_t)G;
    A.width = K * BSA_PAGES_PER_SPARSE_BLOCK;
    A.scale = scale;
    A.status = current_status_word();
    A.out = out;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (D == 64) e = launch_attn_g<2>(A, st);
    else if (D == 128) e = launch_attn_g<4>(A, st);
    else e = launch_attn_g<8>(A, st);
    return e == cudaSuccess ? BSA_OK : (int)e;
}
