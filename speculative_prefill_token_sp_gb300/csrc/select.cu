// Chunk scoring, pooling, chunk selection and position-ID compaction.
//
// Method: paper review "Speculative Prefill ...", chunk formula and section
// "chunk selection and pooling denoising" (chunk means -> 1D average pool ->
// top-K chunks) and "position ID recovery" (kept tokens keep their original
// positions); llama.cpp guide "SpecPrefill -- Implementation Guide", function
// select_chunks (nc = ceil(M/chunk), kc = max(1, ceil(nc * keep_pct)) with a
// float product, ascending output), "v3 Improvements" (structural boost,
// cumulative attention mass) and "v3.1: Score Normalization".
//
// Every result equals the fixed-order fp64 evaluation of the definition --
// token scores left to right inside a chunk, pooled windows left to right, the
// total mass in chunk order and the running mass in ranked order, each step
// rounded to nearest -- bit for bit.  Where a shortcut is taken it is one that
// provably gives that same result: an integer sum where every partial sum of
// the chain is exact, a correctly rounded division by a reciprocal and one
// correction, and a cumulative-mass cut decided from parallel sums only when
// the summation error bound decides it (the chains run otherwise).
//
// Kernels: (0) per-prompt min/max (normalisation only); (1+2) chunk sums and
// means with the pooled scores in one multi-block pass: a warp per chunk for
// plain scores in chunks of up to 64 tokens (chunk_pool_warp_kernel), a thread
// per chunk otherwise (chunk_pool_kernel; each block pools its chunks from a
// shared-memory window with a halo), or chunk sums (1) and a separate pool
// pass (2) for windows wider than the halo; (3) one CTA per prompt: radix
// select of exactly kc chunks on (score desc, index asc) with the keys in
// registers (prompts of up to 4096 chunks; longer ones read them from memory
// each pass), or a bitonic sort of (mean desc, index asc) and the
// running-mass cut; then the exclusive scan of kept chunk sizes and, for
// chunks of up to 256 tokens, the kept positions themselves; (4) compaction of
// the kept positions for larger chunks or longer prompts; (5) the guide's v2
// keep rules (sp_select_rules).
#include "sp_common.cuh"

#include <math.h>
#include <stdint.h>

namespace sp {
namespace {

constexpr int kMaxBatch = 256;
constexpr int kSelThreads = 1024;
constexpr int kRegKeys = 4;             // keys per thread of the in-register top-K (prompts <= 4096 chunks)
constexpr int kInlinePosChunk = 256;    // chunks up to this size get their positions from the selection kernel
constexpr int kMassMaxChunks = 16384;
constexpr int kMaxMinTok = 4096;        // keep-rule minimum, at most
constexpr int kMaxExtras = kMaxMinTok + 6;

struct SelGeo {
    int B, chunk, pool_k;
    int mode;
    double rate;
    int has_boost;
    int first_n, last_n, normalize;
    double first_mult, last_mult;
    double rcp_chunk, rcp_pool;     // RN(1/chunk), RN(1/pool_k) (IEEE division on the host)
    int64_t cu[kMaxBatch + 1];      // token offsets
    int64_t cn[kMaxBatch + 1];      // chunk offsets
    int min_tok, always_keep;       // keep rules (sp_select_rules)
    int64_t max_keep;
};

// IEEE order of doubles as unsigned integers (+0 and -0 map to the same key).
__device__ __forceinline__ uint64_t order_key(double v) {
    if (v == 0.0) v = 0.0;
    uint64_t u = (uint64_t)__double_as_longlong(v);
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// Kernels launched with programmatic stream serialization may start while the
// stream's previous kernel still runs; this waits until that kernel has
// completed and its memory is visible (a no-op after an ordinary launch).
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Prompt offsets from the parameter block.  Reading a parameter array at a
// runtime index is slow on the first touch (microseconds); a single prompt --
// the common call -- reads entries 0 and 1 at fixed offsets instead.
__device__ __forceinline__ int64_t geo_cu(const SelGeo& g, int i) {
    return g.B == 1 ? (i == 0 ? g.cu[0] : g.cu[1]) : g.cu[i];
}
__device__ __forceinline__ int64_t geo_cn(const SelGeo& g, int i) {
    return g.B == 1 ? (i == 0 ? g.cn[0] : g.cn[1]) : g.cn[i];
}

__device__ __forceinline__ int find_batch(const int64_t* cu, int B, int64_t x) {
    int lo = 0, hi = B - 1;                 // largest b with cu[b] <= x
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Offset tables of a batch for kernels that look prompts up by position: the
// B + 1 token and chunk offsets are copied to shared memory once per block (one
// parallel round of parameter reads; a binary search over the parameter block
// would chain its slow reads).  A single prompt keeps the fixed-offset reads.
// Every thread of the block calls stage_tabs before any other use.
struct Tabs {
    const int64_t* cu;
    const int64_t* cn;
};
__device__ __forceinline__ Tabs stage_tabs(const SelGeo& g, int64_t* s_cu, int64_t* s_cn) {
    if (g.B > 1) {
        for (int i = threadIdx.x; i <= g.B; i += blockDim.x) {
            s_cu[i] = g.cu[i];
            s_cn[i] = g.cn[i];
        }
        __syncthreads();
    }
    return {s_cu, s_cn};
}
__device__ __forceinline__ int64_t tab_cu(const SelGeo& g, const Tabs& t, int i) {
    return g.B == 1 ? (i == 0 ? g.cu[0] : g.cu[1]) : t.cu[i];
}
__device__ __forceinline__ int64_t tab_cn(const SelGeo& g, const Tabs& t, int i) {
    return g.B == 1 ? (i == 0 ? g.cn[0] : g.cn[1]) : t.cn[i];
}
__device__ __forceinline__ int chunk_batch(const SelGeo& g, const Tabs& t, int64_t gc) {
    return g.B == 1 ? 0 : find_batch(t.cn, g.B, gc);
}
__device__ __forceinline__ int token_batch(const SelGeo& g, const Tabs& t, int64_t i) {
    return g.B == 1 ? 0 : find_batch(t.cu, g.B, i);
}

// Min-max normalisation of one prompt: x -> (x - mn) / (mx - mn), every score
// 1.0 when mx == mn.  den = mx - mn (one rounding) and rcp = 1 / den (correctly
// rounded) are computed once per prompt.
struct NormCoef {
    double mn, den, rcp;
    int flat;
};

// (0) min and max importance of each prompt (one CTA per prompt).
__global__ void __launch_bounds__(1024) minmax_kernel(const SelGeo g, const float* __restrict__ imp,
                                                      NormCoef* __restrict__ mm, int32_t* __restrict__ hdr) {
    const int b = blockIdx.x;
    const int64_t m0 = geo_cu(g, b), Mb = geo_cu(g, b + 1) - m0;
    wait_prior_grid();
    if (hdr != nullptr && b == 0 && threadIdx.x < (int)(sizeof(WsHeader) / 4)) hdr[threadIdx.x] = 0;
    float mn = INFINITY, mx = -INFINITY;
#pragma unroll 8
    for (int64_t i = threadIdx.x; i < Mb; i += blockDim.x) {
        const float v = imp[m0 + i];
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
    }
    __shared__ float smn[32], smx[32];
    for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if ((threadIdx.x & 31) == 0) { smn[threadIdx.x >> 5] = mn; smx[threadIdx.x >> 5] = mx; }
    __syncthreads();
    if (threadIdx.x < 32) {
        int nw = blockDim.x >> 5;
        mn = threadIdx.x < nw ? smn[threadIdx.x] : INFINITY;
        mx = threadIdx.x < nw ? smx[threadIdx.x] : -INFINITY;
        for (int o = 16; o > 0; o >>= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        if (threadIdx.x == 0) {
            NormCoef c;
            c.flat = mx > mn ? 0 : 1;
            c.mn = (double)mn;
            c.den = __dsub_rn((double)mx, (double)mn);
            c.rcp = c.flat ? 0.0 : __drcp_rn(c.den);
            mm[b] = c;
        }
    }
}

// Token score: fp64 importance, optionally normalised and boosted.
//
// The normalising division (x - mn) / den is correctly rounded without a
// divide instruction (fp64 division is slow on this GPU): with rcp = RN(1/den),
// q0 = RN(num * rcp) is within one ulp of num / den, the residual
// num - q0 * den is exact in one fma, and RN(q0 + residual * rcp) is then the
// correctly rounded quotient (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990).  No step underflows here: num and den are differences of fp32 values.
__device__ __forceinline__ double token_score(const SelGeo& g, float v, int64_t i, int64_t Mb,
                                              const NormCoef& nc) {
    double x = (double)v;
    if (g.has_boost) {
        if (g.normalize) {
            if (!nc.flat) {
                const double num = __dsub_rn(x, nc.mn);
                const double q0 = __dmul_rn(num, nc.rcp);
                const double r = __fma_rn(-q0, nc.den, num);
                x = __fma_rn(r, nc.rcp, q0);
            } else {
                x = 1.0;
            }
        }
        if (i < (int64_t)g.first_n) x = __dmul_rn(x, g.first_mult);
        if (i >= Mb - (int64_t)g.last_n) x = __dmul_rn(x, g.last_mult);
    }
    return x;
}

// RN(s / n) for a count n, with rcp = RN(1/n): q0 = RN(s * rcp) is within one
// ulp of the quotient, the residual s - q0 * n is exact in one fma, and
// RN(q0 + residual * rcp) is the correctly rounded quotient (Markstein's
// theorem, as in token_score).  s is finite here and a sum of fp32 values or of
// their means, so nothing underflows; otherwise the divide instruction.
__device__ __forceinline__ double div_count(double s, int n, double rcp) {
    if (!isfinite(s)) return __ddiv_rn(s, (double)n);
    const double q0 = __dmul_rn(s, rcp);
    const double r = __fma_rn(-q0, (double)n, s);
    return __fma_rn(r, rcp, q0);
}

// A warp's chunk of n <= 64 plain fp32 scores: lane k holds values k and k + 32
// (0 past n).  Their left-to-right fp64 sum is computed exactly in integers when
// every partial sum of that chain is an fp64 number: all values finite and
// >= 0, 2^q the smallest unit in the last place among the nonzero ones (it
// divides every value), and the exact total below 2^(q + 53).  Every partial
// sum is then a multiple of 2^q between 0 and the total, so each rounded
// addition of the chain is exact and the chain's result is the exact total --
// which integer addition gives in any order, here a warp reduction.  Otherwise
// the chain itself runs (every lane the same, on broadcast values).  Every
// lane returns the sum.
__device__ __forceinline__ void decode_f32(float x, bool& ok, int& e, uint64_t& m) {
    const uint32_t u = __float_as_uint(x);
    const uint32_t be = (u >> 23) & 255u;
    ok = (u >> 31) == 0u && be != 255u;
    e = be ? (int)be - 150 : -149;                         // x = m * 2^e
    m = be ? ((u & 0x7fffffu) | 0x800000u) : (u & 0x7fffffu);
}

__device__ __forceinline__ double warp_chunk_sum(float x0, float x1, int n) {
    bool ok0, ok1;
    int e0, e1;
    uint64_t m0, m1;
    decode_f32(x0, ok0, e0, m0);
    decode_f32(x1, ok1, e1, m1);
    int qmin = min(m0 ? e0 : 1 << 20, m1 ? e1 : 1 << 20);
    int emax = max(m0 ? e0 : -(1 << 20), m1 ? e1 : -(1 << 20));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        qmin = min(qmin, __shfl_xor_sync(0xffffffffu, qmin, o));
        emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
    }
    bool exact = __all_sync(0xffffffffu, ok0 && ok1);
    if (exact && emax < qmin) return 0.0;                  // every value is +0
    exact = exact && emax - qmin <= 29;                    // every term below 2^53
    if (exact) {
        uint64_t S = (m0 ? m0 << (e0 - qmin) : 0ull) + (m1 ? m1 << (e1 - qmin) : 0ull);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
        if ((S >> 53) == 0)
            return __dmul_rn(__ull2double_rn(S), __longlong_as_double((long long)(qmin + 1023) << 52));
    }
    double s = 0.0;
    for (int k = 0; k < n; ++k) {
        const float v = __shfl_sync(0xffffffffu, k < 32 ? x0 : x1, k & 31);
        s = __dadd_rn(s, (double)v);
    }
    return s;
}

// (1) chunk sums (left to right from 0.0) and means (one divide).
// Sum (left to right from 0.0) and mean (one divide) of global chunk gc;
// sixteen loads in flight ahead of the additions.
__device__ __forceinline__ void chunk_sum_mean(const SelGeo& g, const Tabs& tb, const float* __restrict__ imp,
                                               const NormCoef* __restrict__ mm, int64_t gc, double& sum, double& mean) {
    const int b = chunk_batch(g, tb, gc);
    const int64_t c = gc - tab_cn(g, tb, b);
    const int64_t m0 = tab_cu(g, tb, b), Mb = tab_cu(g, tb, b + 1) - m0;
    const int64_t lo = c * g.chunk, hi = min(lo + (int64_t)g.chunk, Mb);
    const int n = (int)(hi - lo);
    NormCoef mmb = {0.0, 0.0, 0.0, 1};
    if (g.has_boost && g.normalize) mmb = mm[b];
    double s = 0.0;
    int64_t i = lo;
    for (; i + 16 <= hi; i += 16) {
        float v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = imp[m0 + i + k];
#pragma unroll
        for (int k = 0; k < 16; ++k) s = __dadd_rn(s, token_score(g, v[k], i + k, Mb, mmb));
    }
    for (; i < hi; ++i) s = __dadd_rn(s, token_score(g, imp[m0 + i], i, Mb, mmb));
    sum = s;
    mean = n == g.chunk ? div_count(s, n, g.rcp_chunk) : __ddiv_rn(s, (double)n);
}

__global__ void chunk_kernel(const SelGeo g, const float* __restrict__ imp, const NormCoef* __restrict__ mm,
                             double* __restrict__ sums, double* __restrict__ means, int32_t* __restrict__ hdr) {
    // a fresh status for the call (the workspace header)
    __shared__ int64_t s_cu[kMaxBatch + 1], s_cn[kMaxBatch + 1];
    const Tabs tb = stage_tabs(g, s_cu, s_cn);
    if (hdr != nullptr && blockIdx.x == 0 && threadIdx.x < (int)(sizeof(WsHeader) / 4)) hdr[threadIdx.x] = 0;
    const int64_t total = tab_cn(g, tb, g.B);
    for (int64_t gc = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; gc < total;
         gc += (int64_t)gridDim.x * blockDim.x)
        chunk_sum_mean(g, tb, imp, mm, gc, sums[gc], means[gc]);
}

// (1+2) chunk sums and means, and the centred pool, for the block's 64 chunks:
// the means of the block's chunks and of r = (pool_k - 1) / 2 chunks on each
// side go to shared memory (the halo's are computed again, with the same
// operations), then each chunk's window, clipped to its own prompt, is summed
// left to right from 0.0 and divided by its count, as in pool_kernel.  The
// block has a thread for each of its 64 + 2r means (rounded up to whole warps),
// so every mean is one thread's single chain of additions.
constexpr int kPoolBlock = 64;
constexpr int kMaxPoolHalo = 224;        // r at most: the window's means fit in 4 KB
__global__ void __launch_bounds__(kPoolBlock + 2 * kMaxPoolHalo) chunk_pool_kernel(const SelGeo g, const float* __restrict__ imp,
                                                                const NormCoef* __restrict__ mm,
                                                                double* __restrict__ sums, double* __restrict__ means,
                                                                double* __restrict__ pooled,
                                                                int32_t* __restrict__ hdr) {
    __shared__ double win[kPoolBlock + 2 * kMaxPoolHalo];
    __shared__ int64_t s_cu[kMaxBatch + 1], s_cn[kMaxBatch + 1];
    const Tabs tb = stage_tabs(g, s_cu, s_cn);
    if (hdr != nullptr && blockIdx.x == 0 && threadIdx.x < (int)(sizeof(WsHeader) / 4)) hdr[threadIdx.x] = 0;
    const int64_t total = tab_cn(g, tb, g.B);
    const int r = (g.pool_k - 1) / 2;
    const int64_t gc0 = (int64_t)blockIdx.x * kPoolBlock;
    for (int w = threadIdx.x; w < kPoolBlock + 2 * r; w += blockDim.x) {
        const int64_t gc = gc0 - r + w;
        if (gc < 0 || gc >= total) continue;
        double sm, mn;
        chunk_sum_mean(g, tb, imp, mm, gc, sm, mn);
        win[w] = mn;
        if (w >= r && w < r + kPoolBlock) {
            sums[gc] = sm;
            means[gc] = mn;
        }
    }
    __syncthreads();
    const int64_t gc = gc0 + threadIdx.x;
    if (threadIdx.x >= kPoolBlock || gc >= total) return;
    const int b = chunk_batch(g, tb, gc);
    const int64_t c = gc - tab_cn(g, tb, b), nc = tab_cn(g, tb, b + 1) - tab_cn(g, tb, b);
    const int64_t lo = c - r < 0 ? 0 : c - r;
    const int64_t hi = c + r > nc - 1 ? nc - 1 : c + r;
    double s = 0.0;
    for (int64_t t = lo; t <= hi; ++t) s = __dadd_rn(s, win[threadIdx.x + r + (t - c)]);
    const int cnt = (int)(hi - lo + 1);
    pooled[gc] = cnt == g.pool_k ? div_count(s, cnt, g.rcp_pool) : __ddiv_rn(s, (double)cnt);
}

// (1+2) for plain fp32 scores (no normalisation or boost) in chunks of up to 64
// tokens: one warp per chunk (one coalesced load, the exact sum of
// warp_chunk_sum), kPoolWarps chunks per block of which the first and last r =
// (pool_k - 1) / 2 are the halo of the block's kPoolWarps - 2r pooled outputs
// (their means are computed again by the neighbouring block, with the same
// operations).  Pooling as in chunk_pool_kernel.  Also clears the status header.
constexpr int kPoolWarps = 32;
constexpr int kMaxWarpPoolHalo = 8;
// kBoost: boosted (and normalised) token scores, which are fp64 and get no
// integer sum.  Their fp64 work is spread so that every warp instruction
// carries 32 lanes: each warp computes its chunk's token scores one token per
// lane into shared memory, then warp 0 runs the 32 chunks' chains, one chunk
// per lane (a warp-wide fp64 instruction costs the same with 1 or 32 lanes).
template <bool kBoost>
__global__ void __launch_bounds__(kPoolWarps * 32) chunk_pool_warp_kernel(const SelGeo g, const float* __restrict__ imp,
                                                                       const NormCoef* __restrict__ mm,
                                                                       double* __restrict__ sums,
                                                                       double* __restrict__ means,
                                                                       double* __restrict__ pooled,
                                                                       int32_t* __restrict__ hdr) {
    __shared__ double win[kPoolWarps];
    __shared__ int64_t s_cu[kMaxBatch + 1], s_cn[kMaxBatch + 1];
    const Tabs tb = stage_tabs(g, s_cu, s_cn);
    wait_prior_grid();
    if (hdr != nullptr && blockIdx.x == 0 && threadIdx.x < (int)(sizeof(WsHeader) / 4)) hdr[threadIdx.x] = 0;
    const int64_t total = tab_cn(g, tb, g.B);
    const int r = (g.pool_k - 1) / 2, outs = kPoolWarps - 2 * r;
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t gc0 = (int64_t)blockIdx.x * outs;
    const int64_t gc = gc0 - r + w;
    if constexpr (!kBoost) {
        if (gc >= 0 && gc < total) {
            const int b = chunk_batch(g, tb, gc);
            const int64_t c = gc - tab_cn(g, tb, b);
            const int64_t t0 = tab_cu(g, tb, b), Mb = tab_cu(g, tb, b + 1) - t0;
            const int64_t lo = c * g.chunk;
            const int n = (int)min((int64_t)g.chunk, Mb - lo);
            const float* src = imp + t0 + lo;
            const float x0 = lane < n ? src[lane] : 0.f;
            const float x1 = lane + 32 < n ? src[lane + 32] : 0.f;
            const double sum = warp_chunk_sum(x0, x1, n);
            const double mean = n == g.chunk ? div_count(sum, n, g.rcp_chunk) : __ddiv_rn(sum, (double)n);
            if (lane == 0) {
                win[w] = mean;
                if (w >= r && w < r + outs) {
                    sums[gc] = sum;
                    means[gc] = mean;
                }
            }
        }
    } else {
        __shared__ double xs[64 * (kPoolWarps + 1)];   // token k of the block's chunk w at k * 33 + w
        if (gc >= 0 && gc < total) {
            const int b = chunk_batch(g, tb, gc);
            const int64_t c = gc - tab_cn(g, tb, b);
            const int64_t t0 = tab_cu(g, tb, b), Mb = tab_cu(g, tb, b + 1) - t0;
            const int64_t lo = c * g.chunk;
            const int n = (int)min((int64_t)g.chunk, Mb - lo);
            const NormCoef mmb = g.normalize ? mm[b] : NormCoef{0.0, 0.0, 0.0, 1};
            if (lane < n) xs[lane * (kPoolWarps + 1) + w] = token_score(g, imp[t0 + lo + lane], lo + lane, Mb, mmb);
            if (lane + 32 < n)
                xs[(lane + 32) * (kPoolWarps + 1) + w] = token_score(g, imp[t0 + lo + lane + 32], lo + lane + 32, Mb, mmb);
        }
        __syncthreads();
        if (w == 0) {
            const int64_t gcl = gc0 - r + lane;            // lane c chains the block's chunk c
            if (gcl >= 0 && gcl < total) {
                const int b = chunk_batch(g, tb, gcl);
                const int64_t c = gcl - tab_cn(g, tb, b);
                const int64_t Mb = tab_cu(g, tb, b + 1) - tab_cu(g, tb, b);
                const int n = (int)min((int64_t)g.chunk, Mb - c * g.chunk);
                double sum = 0.0;
                for (int k = 0; k < n; ++k) sum = __dadd_rn(sum, xs[k * (kPoolWarps + 1) + lane]);
                const double mean = n == g.chunk ? div_count(sum, n, g.rcp_chunk) : __ddiv_rn(sum, (double)n);
                win[lane] = mean;
                if (lane >= r && lane < r + outs) {
                    sums[gcl] = sum;
                    means[gcl] = mean;
                }
            }
        }
    }
    if (g.pool_k <= 1) return;
    __syncthreads();
    const int t = threadIdx.x;
    const int64_t gp = gc0 + t;
    if (t >= outs || gp >= total) return;
    const int b = chunk_batch(g, tb, gp);
    const int64_t c = gp - tab_cn(g, tb, b), nc = tab_cn(g, tb, b + 1) - tab_cn(g, tb, b);
    const int64_t lo = c - r < 0 ? 0 : c - r;
    const int64_t hi = c + r > nc - 1 ? nc - 1 : c + r;
    double s = 0.0;
    for (int64_t k = lo; k <= hi; ++k) s = __dadd_rn(s, win[t + r + (k - c)]);
    const int cnt = (int)(hi - lo + 1);
    pooled[gp] = cnt == g.pool_k ? div_count(s, cnt, g.rcp_pool) : __ddiv_rn(s, (double)cnt);
}

// (2) centred average pool over the prompt's own chunks; edges average in-range
// chunks (left to right from 0.0, one divide by the window's count).
__device__ __forceinline__ double pooled_at(const SelGeo& g, const double* __restrict__ means, int64_t c0, int64_t nc,
                                            int64_t c) {
    const int r = (g.pool_k - 1) / 2;
    const int64_t lo = c - r < 0 ? 0 : c - r;
    const int64_t hi = c + r > nc - 1 ? nc - 1 : c + r;
    double s = 0.0;
    for (int64_t t = lo; t <= hi; ++t) s = __dadd_rn(s, means[c0 + t]);
    const int cnt = (int)(hi - lo + 1);
    return cnt == g.pool_k ? div_count(s, cnt, g.rcp_pool) : __ddiv_rn(s, (double)cnt);
}

__global__ void pool_kernel(const SelGeo g, const double* __restrict__ means, double* __restrict__ pooled) {
    __shared__ int64_t s_cu[kMaxBatch + 1], s_cn[kMaxBatch + 1];
    const Tabs tb = stage_tabs(g, s_cu, s_cn);
    const int64_t total = tab_cn(g, tb, g.B);
    for (int64_t gc = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; gc < total;
         gc += (int64_t)gridDim.x * blockDim.x) {
        const int b = chunk_batch(g, tb, gc);
        const int64_t c0 = tab_cn(g, tb, b), nc = tab_cn(g, tb, b + 1) - c0;
        pooled[gc] = pooled_at(g, means, c0, nc, gc - c0);
    }
}

// Block-wide exclusive scan of one 64-bit value per thread; returns the prefix
// and writes the block total to *total (all threads).
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* sh, long long* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    long long x = v;
    for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[w] = x;
    __syncthreads();
    if (w == 0) {
        long long s = lane < nw ? sh[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            long long y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < nw) sh[lane] = s;             // inclusive warp totals
    }
    __syncthreads();
    long long base = w > 0 ? sh[w - 1] : 0;
    *total = sh[nw - 1];
    __syncthreads();
    return base + x - v;
}

// The same for 32-bit values (half the shuffles).
__device__ __forceinline__ int block_exclusive_scan32(int v, int* sh, int* total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[w] = x;
    __syncthreads();
    if (w == 0) {
        int s = lane < nw ? sh[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < nw) sh[lane] = s;
    }
    __syncthreads();
    const int base = w > 0 ? sh[w - 1] : 0;
    *total = sh[nw - 1];
    __syncthreads();
    return base + x - v;
}

// Top-K of a prompt with at most kSelThreads * kRegKeys chunks: the pooled keys
// (chunk c = q * blockDim.x + tid in key[q]) stay in registers through a radix
// select, 8 bits per pass from the most significant, counted with
// warp-aggregated shared-memory atomics.  The passes stop once every key with
// the selected prefix is taken.  Then keys above the prefix, and the first
// `remaining` equal to it in chunk order, are kept.
__device__ __forceinline__ void topk_in_registers(const SelGeo& g, const double* __restrict__ keys_src, int64_t c0, int nc, int64_t Mb,
                                  int kc, int* __restrict__ flags, int64_t* __restrict__ offs,
                                  int32_t* __restrict__ kept_b, int64_t* __restrict__ n_kept_b, unsigned* hist,
                                  long long* scan_sh, int* scan32, uint64_t* s_prefix, int* s_remaining, int* s_done) {
    const int tid = threadIdx.x, lane = tid & 31, bd = blockDim.x;
    const int rounds = (nc + bd - 1) / bd;
    uint64_t key[kRegKeys];
#pragma unroll
    for (int q = 0; q < kRegKeys; ++q) {
        const int c = q * bd + tid;
        key[q] = c < nc ? order_key(keys_src[c0 + c]) : 0ull;
    }
    uint64_t prefix = 0, pmask = 0;
    int remaining = kc;
    bool done = false;                     // every key equal to the prefix is taken
    for (int pass = 0; pass < 8; ++pass) {
        const int shift = 56 - 8 * pass;
        for (int i = tid; i < 256; i += bd) hist[i] = 0;
        if (tid == 0) *s_done = 0;
        __syncthreads();
#pragma unroll
        for (int q = 0; q < kRegKeys; ++q) {
            if (q >= rounds) break;
            const int c = q * bd + tid;
            const bool take = c < nc && (key[q] & pmask) == prefix;
            const unsigned digit = take ? (unsigned)((key[q] >> shift) & 255u) : 256u;
            const unsigned peers = __match_any_sync(0xffffffffu, digit);
            if (take && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], (unsigned)__popc(peers));
        }
        __syncthreads();
        if (tid < 32) {
            // lane covers digits [8*lane, 8*lane+8); count keys with a larger digit.
            unsigned local = 0;
            for (int q = 0; q < 8; ++q) local += hist[tid * 8 + q];
            unsigned x = local;
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_down_sync(0xffffffffu, x, o);
                if (tid + o < 32) x += y;
            }
            const unsigned above = x - local;
            if (above < (unsigned)remaining && above + local >= (unsigned)remaining) {
                unsigned cum = above;
                for (int q = 7; q >= 0; --q) {
                    const unsigned hq = hist[tid * 8 + q];
                    if (cum + hq >= (unsigned)remaining) {
                        *s_prefix = prefix | ((uint64_t)(tid * 8 + q) << shift);
                        *s_remaining = remaining - (int)cum;
                        *s_done = hq == (unsigned)(remaining - (int)cum) ? 1 : 0;
                        break;
                    }
                    cum += hq;
                }
            }
        }
        __syncthreads();
        prefix = *s_prefix;
        remaining = *s_remaining;
        pmask |= (0xFFull << shift);
        done = *s_done != 0;
        __syncthreads();
        if (done) break;
    }
    // Keys above the prefix are kept, and the first `remaining` equal to it in
    // chunk order -- all of them when the last pass found exactly that many,
    // which needs no ranking scan.  Output offsets: an exclusive scan of the
    // kept chunk sizes (32-bit while the prompt is below 2^31 tokens).  Each
    // warp then writes its kept chunks' positions together, one chunk at a
    // time, lanes over the chunk's tokens.
    const bool narrow = Mb < (int64_t)INT32_MAX;
    const bool inline_pos = g.chunk <= kInlinePosChunk;
    long long taken_eq = 0, running = 0;
#pragma unroll
    for (int q = 0; q < kRegKeys; ++q) {
        if (q >= rounds) break;
        const int c = q * bd + tid;
        const bool in = c < nc;
        const uint64_t k = key[q] & pmask;
        const bool gt = in && k > prefix, eq = in && k == prefix;
        bool keep = gt || eq;
        if (!done) {
            long long tot_eq;
            const long long rank = block_exclusive_scan(eq ? 1 : 0, scan_sh, &tot_eq);
            keep = gt || (eq && taken_eq + rank < remaining);
            taken_eq += tot_eq;
        }
        const int64_t lo = (int64_t)c * g.chunk;
        const long long sz = keep ? (long long)(min(lo + (int64_t)g.chunk, Mb) - lo) : 0;
        long long off, tot_sz;
        if (narrow) {
            int t32;
            off = block_exclusive_scan32((int)sz, scan32, &t32);
            tot_sz = t32;
        } else {
            off = block_exclusive_scan(sz, scan_sh, &tot_sz);
        }
        if (in) {
            flags[c0 + c] = keep ? 1 : 0;
            offs[c0 + c] = running + off;
        }
        if (inline_pos) {
            unsigned kb = __ballot_sync(0xffffffffu, keep);
            while (kb) {
                const int src = __ffs(kb) - 1;
                kb &= kb - 1;
                const long long o = __shfl_sync(0xffffffffu, running + off, src);
                const long long l = __shfl_sync(0xffffffffu, (long long)lo, src);
                const int n = __shfl_sync(0xffffffffu, (int)sz, src);
                for (int t = lane; t < n; t += 32) kept_b[o + t] = (int32_t)(l + t);
            }
        }
        running += tot_sz;
    }
    if (tid == 0) *n_kept_b = running;
}

// (3) per-prompt selection.  Writes keep flags, kept-size offsets and n_kept.
// (one instantiation per mode: each launch carries only its mode's code)
template <int kMode>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelGeo g, const double* __restrict__ sums,
                                                             const double* __restrict__ means,
                                                             const double* __restrict__ pooled,
                                                             int* __restrict__ flags,
                                                             int64_t* __restrict__ offs,
                                                             int32_t* __restrict__ kept_pos,
                                                             int64_t* __restrict__ n_kept) {
    extern __shared__ __align__(16) unsigned char dsm[];
    __shared__ long long scan_sh[32];
    __shared__ int scan32[32];
    __shared__ unsigned hist[256];
    __shared__ uint64_t s_prefix;
    __shared__ int s_remaining;
    __shared__ int s_kstar;
    __shared__ int s_done;
    __shared__ int s_flag[32];
    __shared__ double s_rhs[2];
    __shared__ double s_block[64];

    const int b = blockIdx.x;
    const int64_t c0 = geo_cn(g, b);
    const int nc = (int)(geo_cn(g, b + 1) - c0);
    const int64_t Mb = geo_cu(g, b + 1) - geo_cu(g, b);
    const int tid = threadIdx.x;
    wait_prior_grid();
    if (nc == 0) {
        if (tid == 0) n_kept[b] = 0;
        return;
    }

    if constexpr (kMode == SP_SELECT_TOPK) {
        // kc = max(1, ceil(f32(nc) * f32(keep_rate))), at most nc.
        const float prod = (float)nc * (float)g.rate;
        int kc = (int)ceilf(prod);
        kc = kc < 1 ? 1 : (kc > nc ? nc : kc);
        if (nc <= (int)blockDim.x * kRegKeys) {
            topk_in_registers(g, g.pool_k > 1 ? pooled : means, c0, nc, Mb, kc, flags, offs, kept_pos + geo_cu(g, b),
                              n_kept + b, hist, scan_sh, scan32,
                              &s_prefix, &s_remaining, &s_done);
            return;
        }
        // Radix select (8 bits per pass, most significant first) of the kc-th
        // largest key; afterwards `remaining` keys equal to it must be taken.
        uint64_t prefix = 0, pmask = 0;
        int remaining = kc;
        for (int pass = 0; pass < 8; ++pass) {
            const int shift = 56 - 8 * pass;
            for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
            __syncthreads();
            for (int c = tid; c < nc; c += blockDim.x) {
                uint64_t k = order_key(pooled[c0 + c]);
                if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (tid < 32) {
                // lane covers digits [8*lane, 8*lane+8); count keys with a larger digit.
                unsigned local = 0;
                for (int q = 0; q < 8; ++q) local += hist[tid * 8 + q];
                unsigned above = 0;                   // sum over lanes > tid
                unsigned x = local;
                for (int o = 1; o < 32; o <<= 1) {
                    unsigned y = __shfl_down_sync(0xffffffffu, x, o);
                    if (tid + o < 32) x += y;
                }
                above = x - local;                    // inclusive suffix minus own
                if (above < (unsigned)remaining && above + local >= (unsigned)remaining) {
                    unsigned cum = above;
                    for (int q = 7; q >= 0; --q) {
                        unsigned hq = hist[tid * 8 + q];
                        if (cum + hq >= (unsigned)remaining) {
                            s_prefix = prefix | ((uint64_t)(tid * 8 + q) << shift);
                            s_remaining = remaining - (int)cum;
                            break;
                        }
                        cum += hq;
                    }
                }
            }
            __syncthreads();
            prefix = s_prefix;
            remaining = s_remaining;
            pmask |= (0xFFull << shift);
            __syncthreads();
        }
        const uint64_t T = prefix;
        long long taken_eq = 0, running = 0;
        for (int base = 0; base < nc; base += blockDim.x) {
            const int c = base + tid;
            const bool in = c < nc;
            const uint64_t k = in ? order_key(pooled[c0 + c]) : 0;
            const bool gt = in && k > T, eq = in && k == T;
            long long tot_eq;
            long long rank = block_exclusive_scan(eq ? 1 : 0, scan_sh, &tot_eq);
            const bool keep = gt || (eq && taken_eq + rank < remaining);
            const int64_t lo = (int64_t)c * g.chunk;
            const long long sz = keep ? (long long)(min(lo + (int64_t)g.chunk, Mb) - lo) : 0;
            long long tot_sz;
            long long off = block_exclusive_scan(sz, scan_sh, &tot_sz);
            if (in) {
                flags[c0 + c] = keep ? 1 : 0;
                offs[c0 + c] = running + off;
            }
            taken_eq += tot_eq;
            running += tot_sz;
        }
        if (tid == 0) n_kept[b] = running;
        return;
    }

    // Cumulative-mass mode: rank the chunks (descending mean, then index) and
    // keep the shortest ranked prefix whose running mass R_k, added in ranked
    // order, reaches target = RN(tau * total), the total added in chunk order
    // (both chains in fp64, left to right).  The two chains are not run.
    // With every chunk sum finite and >= 0, each chain's result is within
    // gamma_n = n u / (1 - n u) (u = 2^-53) relative of its exact sum (the
    // error bound of recursive summation), and a tree sum or a parallel
    // prefix sum is within gamma_L of it for its depth L <= 64.  So with
    // E = (nc + 80) 2^-52, which covers both and the roundings of the test
    // itself, the prefix sum P_k and total P_n from the parallel sums decide
    //   R_k >= target  when P_k (1 - E) > tau P_n (1 + E),
    //   R_k <  target  when P_k (1 + E) < tau P_n (1 - E).
    // The cut is the first k not decided "below"; if that one is not decided
    // "reached", or a sum is negative or not finite, the two chains run
    // serially, exactly as defined.
    int P = 1;
    while (P < nc) P <<= 1;
    uint64_t* keys = reinterpret_cast<uint64_t*>(dsm);
    int* idx = reinterpret_cast<int*>(dsm + sizeof(uint64_t) * P);
    double* ranked = reinterpret_cast<double*>(keys);
    const int nt = (int)blockDim.x, lane = tid & 31, wid = tid >> 5;
    // sort keys, and the check that every chunk sum is finite and >= 0 (its
    // bits below those of +inf); fp64 work is kept to the threads that need it,
    // fp64 throughput being low on this GPU
    bool fine = true;
    for (int i = tid; i < P; i += nt) {
        if (i < nc) {
            keys[i] = ~order_key(means[c0 + i]);
            idx[i] = i;
            fine = fine && (uint64_t)__double_as_longlong(sums[c0 + i]) < 0x7ff0000000000000ull;
        } else {
            keys[i] = ~0ull;
            idx[i] = 0x7fffffff;
        }
    }
    fine = __all_sync(0xffffffffu, fine);
    if (lane == 0) s_flag[wid] = fine ? 1 : 0;
    if (tid == 0) { s_kstar = nc; s_done = 0; }
    __syncthreads();
    if (P <= nt) {
        // one (key, index) per thread: bitonic stages with partners inside the
        // warp by shuffles, the others through shared memory
        uint64_t k = tid < P ? keys[tid] : ~0ull;
        int x = tid < P ? idx[tid] : 0x7fffffff;
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                uint64_t kp;
                int xp;
                if (stride >= 32) {
                    __syncthreads();
                    if (tid < P) { keys[tid] = k; idx[tid] = x; }
                    __syncthreads();
                    kp = tid < P ? keys[tid ^ stride] : ~0ull;
                    xp = tid < P ? idx[tid ^ stride] : 0x7fffffff;
                } else {
                    kp = __shfl_xor_sync(0xffffffffu, k, stride);
                    xp = __shfl_xor_sync(0xffffffffu, x, stride);
                }
                // ascending within blocks of `size` whose bit `size` is 0, descending in the others;
                // the lower thread of a pair keeps the smaller in an ascending block
                const bool up = (tid & size) == 0, lower = (tid & stride) == 0;
                const bool mine_gt = k > kp || (k == kp && x > xp);
                if (mine_gt == (up == lower)) { k = kp; x = xp; }
            }
        }
        __syncthreads();
        if (tid < P) { keys[tid] = k; idx[tid] = x; }
    } else {
        for (int size = 2; size <= P; size <<= 1) {
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < P / 2; i += nt) {
                    const int lo = 2 * i - (i & (stride - 1));
                    const int hi = lo + stride;
                    const bool up = (lo & size) == 0;
                    const uint64_t ka = keys[lo], kb = keys[hi];
                    const int ia = idx[lo], ib = idx[hi];
                    const bool a_gt_b = ka > kb || (ka == kb && ia > ib);
                    if (a_gt_b == up) {
                        keys[lo] = kb; keys[hi] = ka;
                        idx[lo] = ib; idx[hi] = ia;
                    }
                }
                __syncthreads();
            }
        }
    }
    __syncthreads();
    bool all_fine = true;
    for (int w = 0; w < nt / 32; ++w) all_fine = all_fine && s_flag[w] != 0;
    // prefix sums in ranked order: a contiguous segment per thread, a scan of
    // the segment totals inside each warp that holds chunks, then across those
    // warps; the last prefix is the total
    const int seg = (nc + nt - 1) / nt, k0 = tid * seg, k1 = min(k0 + seg, nc);
    const int wact = (nc + 32 * seg - 1) / (32 * seg);   // warps that hold chunks
    double loc = 0.0, incl = 0.0;
    if (wid < wact) {
        for (int k = k0; k < k1; ++k) {
            const double v = sums[c0 + idx[k]];
            loc = k == k0 ? v : __dadd_rn(loc, v);
        }
        incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl = __dadd_rn(incl, y);
        }
        if (lane == 31) s_block[wid] = incl;
    }
    __syncthreads();
    if (wid == 0) {
        double w_in = lane < wact ? s_block[lane] : 0.0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, w_in, o);
            if (lane >= o) w_in = __dadd_rn(w_in, y);
        }
        s_block[32 + lane] = w_in;                     // inclusive over warps
    }
    __syncthreads();
    const double E = (double)(nc + 80) * 0x1p-52;
    if (tid == 0) {
        const double total_c = s_block[32 + wact - 1];
        s_rhs[0] = __dmul_rn(__dmul_rn(g.rate, total_c), 1.0 + E);
        s_rhs[1] = __dmul_rn(__dmul_rn(g.rate, total_c), 1.0 - E);
    }
    __syncthreads();
    const double rhs_hi = s_rhs[0], rhs_lo = s_rhs[1];
    if (wid < wact) {
        // the exclusive prefix of this thread's segment: the warps before, then the lanes before
        const double lanes_before = __shfl_up_sync(0xffffffffu, incl, 1);
        double run = wid > 0 ? s_block[32 + wid - 1] : 0.0;
        if (lane > 0) run = wid > 0 ? __dadd_rn(run, lanes_before) : lanes_before;
        for (int k = k0; k < k1; ++k) {
            const double v = sums[c0 + idx[k]];
            run = (k == 0) ? v : __dadd_rn(run, v);
            ranked[k] = run;                           // P_k, the prefix through position k
            const bool below = __dmul_rn(run, 1.0 + E) < rhs_lo;
            if (!below) {
                atomicMin(&s_kstar, k);
                break;
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        const int ka = s_kstar;                        // first position not decided "below"
        bool decided = all_fine;
        if (decided && ka < nc) decided = __dmul_rn(ranked[ka], 1.0 - E) > rhs_hi;
        s_kstar = ka < nc ? ka + 1 : nc;
        s_done = decided ? 0 : 1;                      // 1: run the chains
    }
    __syncthreads();
    if (s_done) {
        // the definition itself: the total in chunk order, then the running
        // mass in ranked order, one thread
        if (tid == 0) {
            double total = 0.0;
            for (int c = 0; c < nc; ++c) total = __dadd_rn(total, sums[c0 + c]);
            const double target = __dmul_rn(g.rate, total);
            double cum = 0.0;
            int kstar = nc;
            for (int k = 0; k < nc; ++k) {
                cum = __dadd_rn(cum, sums[c0 + idx[k]]);
                if (cum >= target) {
                    kstar = k + 1;
                    break;
                }
            }
            s_kstar = kstar;
        }
        __syncthreads();
    }
    const int kstar = s_kstar;
    // the kept flags also in shared memory (over the ranked prefixes, no longer needed)
    int* kept_sh = reinterpret_cast<int*>(keys);
    for (int k = tid; k < nc; k += nt) {
        const int c = idx[k], f = k < kstar ? 1 : 0;
        kept_sh[c] = f;
        flags[c0 + c] = f;
    }
    __syncthreads();
    const bool narrow = Mb < (int64_t)INT32_MAX;
    long long running = 0;
    for (int base = 0; base < nc; base += nt) {
        const int c = base + tid;
        const bool in = c < nc;
        const bool keep = in && kept_sh[c] != 0;
        const int64_t lo = (int64_t)c * g.chunk;
        const long long sz = keep ? (long long)(min(lo + (int64_t)g.chunk, Mb) - lo) : 0;
        long long off, tot_sz;
        if (narrow) {
            int t32;
            off = block_exclusive_scan32((int)sz, scan32, &t32);
            tot_sz = t32;
        } else {
            off = block_exclusive_scan(sz, scan_sh, &tot_sz);
        }
        if (in) offs[c0 + c] = running + off;
        if (g.chunk <= kInlinePosChunk) {
            unsigned kb = __ballot_sync(0xffffffffu, keep);
            while (kb) {
                const int src = __ffs(kb) - 1;
                kb &= kb - 1;
                const long long o = __shfl_sync(0xffffffffu, running + off, src);
                const long long l = __shfl_sync(0xffffffffu, (long long)lo, src);
                const int n = __shfl_sync(0xffffffffu, (int)sz, src);
                for (int t = lane; t < n; t += 32) kept_pos[geo_cu(g, b) + o + t] = (int32_t)(l + t);
            }
        }
        running += tot_sz;
    }
    if (tid == 0) n_kept[b] = running;
}

// (4) every token of a kept chunk writes its original position.
__global__ void compact_kernel(const SelGeo g, const int* __restrict__ flags,
                               const int64_t* __restrict__ offs, int32_t* __restrict__ kept_pos) {
    __shared__ int64_t s_cu[kMaxBatch + 1], s_cn[kMaxBatch + 1];
    const Tabs tb = stage_tabs(g, s_cu, s_cn);
    const int64_t T = tab_cu(g, tb, g.B);
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < T;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int b = token_batch(g, tb, t);
        const int64_t m0 = tab_cu(g, tb, b), i = t - m0, c = i / g.chunk;
        const int64_t gc = tab_cn(g, tb, b) + c;
        if (flags[gc]) kept_pos[m0 + offs[gc] + (i - c * g.chunk)] = (int32_t)i;
    }
}

// (5) the guide's v2 keep rules on one prompt's selection (llama.cpp guide,
// "Full Source Code": select_chunks' always-kept tokens and minimum-token
// back-fill, the main program's SP_MAX_KEEP cap), one block per prompt:
//   eff_min = min(min_tok, max(4, M / 10)); M <= eff_min keeps every token;
//   always_keep adds tokens 0..3 and, if M > 4, M-2 and M-1;
//   while fewer than eff_min are kept, tokens of unselected chunks join in
//   chunk, then token order; the result is ascending;
//   more than max_keep (> 0): every (n / max_keep)-th token, at most max_keep,
//   the last replaced by the last kept token.
__global__ void __launch_bounds__(1024) rules_kernel(const SelGeo g, const int* __restrict__ flags,
                                                     int32_t* __restrict__ kept_pos, int64_t* __restrict__ n_kept,
                                                     int32_t* __restrict__ scratch) {
    __shared__ int32_t extra[kMaxExtras];
    __shared__ int n_extra;
    __shared__ int64_t total_sh;
    const int b = blockIdx.x;
    const int64_t m0 = geo_cu(g, b), M = geo_cu(g, b + 1) - m0;
    const int64_t c0 = geo_cn(g, b), nc = geo_cn(g, b + 1) - c0;
    int32_t* kept = kept_pos + m0;
    int32_t* S = scratch + m0;                   // merged list
    const int64_t n = n_kept[b];
    const int64_t eff_min = g.min_tok > 0 ? min((int64_t)g.min_tok, max((int64_t)4, M / 10)) : 0;
    if (M == 0) return;
    if (M <= eff_min) {
        for (int64_t i = threadIdx.x; i < M; i += blockDim.x) S[i] = (int32_t)i;
        if (threadIdx.x == 0) total_sh = M;
    } else {
        if (threadIdx.x == 0) {
            // tokens to add, ascending: always-kept ones outside kept chunks, then the
            // back-fill (distinct from kept tokens by construction, and checked
            // against the always-kept ones)
            int32_t always[6];
            int na = 0;
            if (g.always_keep) {
                const int64_t cand[6] = {0, 1, 2, 3, M - 2, M - 1};
                const int nc6 = M > 4 ? 6 : 4;
                for (int k = 0; k < nc6; ++k) {
                    const int64_t a = cand[k];
                    if (a < M && !flags[c0 + a / g.chunk]) always[na++] = (int32_t)a;
                }
            }
            int64_t have = n + na;
            int m = 0;
            for (int64_t c = 0; c < nc && have < eff_min; ++c) {
                if (flags[c0 + c]) continue;
                const int64_t e = min((c + 1) * (int64_t)g.chunk, M);
                for (int64_t i = c * g.chunk; i < e && have < eff_min; ++i) {
                    bool dup = false;
                    for (int k = 0; k < na; ++k) dup |= always[k] == (int32_t)i;
                    if (!dup) { extra[m++] = (int32_t)i; ++have; }
                }
            }
            // insert the always-kept tokens into the ascending back-fill list
            for (int k = 0; k < na; ++k) {
                int pos = m++;
                while (pos > 0 && extra[pos - 1] > always[k]) { extra[pos] = extra[pos - 1]; --pos; }
                extra[pos] = always[k];
            }
            n_extra = m;
            total_sh = n + m;
        }
        __syncthreads();
        const int m = n_extra;
        // merge: a kept token moves right by the extras below it, an extra by the kept tokens below it
        for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
            const int32_t v = kept[i];
            int lo = 0, hi = m;
            while (lo < hi) { const int mid = (lo + hi) >> 1; if (extra[mid] < v) lo = mid + 1; else hi = mid; }
            S[i + lo] = v;
        }
        for (int k = threadIdx.x; k < m; k += blockDim.x) {
            const int32_t v = extra[k];
            int64_t lo = 0, hi = n;
            while (lo < hi) { const int64_t mid = (lo + hi) >> 1; if (kept[mid] < v) lo = mid + 1; else hi = mid; }
            S[k + lo] = v;
        }
    }
    __syncthreads();
    const int64_t total = total_sh;
    if (g.max_keep > 0 && total > g.max_keep) {
        const int64_t step = total / g.max_keep;
        const int64_t cnt = min(g.max_keep, (total + step - 1) / step);
        for (int64_t k = threadIdx.x; k < cnt; k += blockDim.x) kept[k] = S[k * step];
        __syncthreads();
        if (threadIdx.x == 0) {
            if (kept[cnt - 1] != S[total - 1]) kept[cnt - 1] = S[total - 1];
            n_kept[b] = cnt;
        }
    } else {
        for (int64_t k = threadIdx.x; k < total; k += blockDim.x) kept[k] = S[k];
        if (threadIdx.x == 0) n_kept[b] = total;
    }
}

struct SelLayout {
    size_t mm, sums, means, pooled, flags, offs, scratch, total;
};

SelLayout sel_layout(const SelectProblem& p) {
    Carve c;
    SelLayout lo;
    const size_t nc = (size_t)std::max<int64_t>(p.total_chunks, 1);
    lo.mm = c.take(sizeof(NormCoef) * std::max(p.B, 1));
    lo.sums = c.take(sizeof(double) * nc);
    lo.means = c.take(sizeof(double) * nc);
    lo.pooled = c.take(sizeof(double) * nc);
    lo.flags = c.take(sizeof(int) * nc);
    lo.offs = c.take(sizeof(int64_t) * nc);
    lo.scratch = p.has_rules ? c.take(sizeof(int32_t) * (size_t)std::max<int64_t>(p.T, 1)) : c.off;
    lo.total = c.off;
    return lo;
}

}  // namespace

size_t select_ws_bytes(const SelectProblem& p) { return sel_layout(p).total; }

namespace {
// A launch that may be scheduled while the stream's previous kernel still runs
// (programmatic stream serialization); the kernel waits for that kernel with
// wait_prior_grid() before it reads or writes memory.  It hides the launch and
// the block start-up behind the previous kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_early(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t st,
                         Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
}  // namespace

sp_status select_launch(const SelectProblem& p, void* ws, cudaStream_t st) {
    if (p.B > kMaxBatch) {
        set_error("sp_select: batch of %d prompts exceeds the supported %d", p.B, kMaxBatch);
        return SP_EUNSUPPORTED;
    }
    if (p.mode == SP_SELECT_MASS && p.max_nc > kMassMaxChunks) {
        set_error("sp_select: cumulative-mass mode supports at most %d chunks per prompt (got %lld)",
                  kMassMaxChunks, (long long)p.max_nc);
        return SP_EUNSUPPORTED;
    }
    SelGeo g;
    g.B = p.B; g.chunk = p.chunk; g.pool_k = p.pool_k; g.mode = (int)p.mode; g.rate = p.rate;
    g.has_boost = p.has_boost ? 1 : 0;
    g.first_n = p.boost.first_n; g.last_n = p.boost.last_n; g.normalize = p.boost.normalize;
    g.first_mult = p.boost.first_mult; g.last_mult = p.boost.last_mult;
    g.rcp_chunk = 1.0 / (double)p.chunk;
    g.rcp_pool = 1.0 / (double)p.pool_k;
    g.min_tok = p.has_rules ? p.rules.min_tok : 0;
    g.always_keep = p.has_rules ? p.rules.always_keep : 0;
    g.max_keep = p.has_rules ? p.rules.max_keep : 0;
    g.cu[0] = 0; g.cn[0] = 0;
    for (int b = 0; b < p.B; ++b) {
        g.cu[b + 1] = p.cu_M_host[b + 1];
        const int64_t Mb = p.cu_M_host[b + 1] - p.cu_M_host[b];
        g.cn[b + 1] = g.cn[b] + (Mb + p.chunk - 1) / p.chunk;
    }
    g.cu[0] = p.cu_M_host[0];
    const SelLayout lo = sel_layout(p);
    char* w = static_cast<char*>(ws);
    NormCoef* mm = reinterpret_cast<NormCoef*>(w + lo.mm);
    double* sums = reinterpret_cast<double*>(w + lo.sums);
    double* means = reinterpret_cast<double*>(w + lo.means);
    double* pooled = reinterpret_cast<double*>(w + lo.pooled);
    int* flags = reinterpret_cast<int*>(w + lo.flags);
    int64_t* offs = reinterpret_cast<int64_t*>(w + lo.offs);

    const int64_t total = g.cn[p.B];
    // the header is cleared by the min/max kernel or the chunk kernel (or here,
    // when there are no chunks)
    const bool normalize = p.has_boost && p.boost.normalize;
    if (total == 0) SP_CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(WsHeader), st));
    if (normalize && total > 0) {
        SP_CUDA_TRY(launch_early(minmax_kernel, (unsigned)p.B, 1024, 0, st, g, p.importance, mm,
                                 static_cast<int32_t*>(ws)));
        SP_LAUNCH_CHECK();
    }
    if (total > 0) {
        // small blocks: the fixed-order fp64 sums run on as many SMs as possible
        int32_t* hdr = normalize ? nullptr : static_cast<int32_t*>(ws);
        const bool pool = p.mode == SP_SELECT_TOPK && p.pool_k > 1;
        const int r = pool ? (p.pool_k - 1) / 2 : 0;
        if (p.chunk <= 64 && r <= kMaxWarpPoolHalo) {
            // chunks of up to 64 tokens: a warp per chunk
            SelGeo gw = g;
            if (!pool) gw.pool_k = 1;
            const int outs = kPoolWarps - 2 * r;
            auto* kern = p.has_boost ? chunk_pool_warp_kernel<true> : chunk_pool_warp_kernel<false>;
            SP_CUDA_TRY(launch_early(kern, (unsigned)((total + outs - 1) / outs), kPoolWarps * 32, 0, st, gw,
                                     p.importance, (const NormCoef*)mm, sums, means, pooled, hdr));
            SP_LAUNCH_CHECK();
        } else if (pool && (p.pool_k - 1) / 2 <= kMaxPoolHalo) {
            const int threads = (kPoolBlock + (p.pool_k - 1) + 31) / 32 * 32;     // 64 + 2r means, whole warps
            chunk_pool_kernel<<<(unsigned)((total + kPoolBlock - 1) / kPoolBlock), threads, 0, st>>>(
                g, p.importance, mm, sums, means, pooled, hdr);
            SP_LAUNCH_CHECK();
        } else {
            const int blocks = (int)std::min<int64_t>((total + 63) / 64, 8192);
            chunk_kernel<<<blocks, 64, 0, st>>>(g, p.importance, mm, sums, means, hdr);
            SP_LAUNCH_CHECK();
            if (pool) {
                pool_kernel<<<(int)std::min<int64_t>((total + 255) / 256, 2048), 256, 0, st>>>(g, means, pooled);
                SP_LAUNCH_CHECK();
            }
        }
    }
    size_t dyn = 0;
    if (p.mode == SP_SELECT_MASS) {
        int P = 1;
        while (P < p.max_nc) P <<= 1;
        dyn = (sizeof(uint64_t) + sizeof(int)) * (size_t)P;
    }
    auto* sel_kern = p.mode == SP_SELECT_MASS ? select_kernel<SP_SELECT_MASS> : select_kernel<SP_SELECT_TOPK>;
    SP_CUDA_TRY(cudaFuncSetAttribute(sel_kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)std::max<size_t>(dyn, 0)));
    SP_CUDA_TRY(launch_early(sel_kern, (unsigned)p.B, kSelThreads, dyn, st, g, (const double*)sums,
                             (const double*)means, (const double*)pooled, flags, offs, p.kept_pos, p.n_kept));
    SP_LAUNCH_CHECK();
    // positions not written by the selection kernel: chunks above kInlinePosChunk
    // tokens, or top-K prompts too long for the in-register path
    const bool inline_pos = p.chunk <= kInlinePosChunk &&
                            (p.mode == SP_SELECT_MASS || p.max_nc <= (int64_t)kSelThreads * kRegKeys);
    if (p.T > 0 && !inline_pos) {
        const int blocks = (int)std::min<int64_t>((p.T + 255) / 256, 4096);
        compact_kernel<<<blocks, 256, 0, st>>>(g, flags, offs, p.kept_pos);
        SP_LAUNCH_CHECK();
    }
    if (p.has_rules && p.T > 0) {
        rules_kernel<<<p.B, 1024, 0, st>>>(g, flags, p.kept_pos, p.n_kept,
                                           reinterpret_cast<int32_t*>(w + lo.scratch));
        SP_LAUNCH_CHECK();
    }
    return SP_OK;
}

}  // namespace sp
