// Look-ahead attention importance, general-shape path (CUDA cores, fp32 FMA).
//
// Covers every shape and dtype the ABI accepts (fp32 or bf16 inputs, any
// d % 8 == 0 up to 256, any N * G rows, ragged batches).  The bf16 shapes the
// tensor-core path handles go there instead; this path is the exact-fp32
// reference-grade implementation used for fp32 inputs and unusual shapes.
//
// Method (paper review "Speculative Prefill ...", core formulas; llama.cpp
// guide "SpecPrefill -- Implementation Guide", Token Importance):
//   s[l,h,j,i] = Q_la[j,l,h] . K[l,g,i] / sqrt(d)            prompt logits
//   lse[l,h,j] = log(sum_i exp(s) + sum_{k<=j} exp(u_k))      u: look-ahead logits
//   acc[j,i]   = max_{l,h} exp(s[l,h,j,i] - lse[l,h,j])
//   importance[i] = (1/N) sum_j acc[j,i]
//
// Kernels: (1) split-S partial softmax statistics (max, sum of exp) per row,
// (2) combine the splits and fold in the causal look-ahead keys -> lse,
// (3) recompute the logits, normalise, max over the heads of the group and
// atomicMax (on the bits of the non-negative weights) across KV heads and
// layers, (4) mean over look-ahead steps.
#include "sp_common.cuh"

#include <math.h>

namespace sp {
namespace {

constexpr int kThreads = 256;
constexpr int kSplit = 256;     // prompt tokens per CTA
constexpr int kSub = 32;        // tokens staged in shared memory at a time
constexpr int kRowsMax = 64;    // rows (look-ahead step x head of the group) per CTA
constexpr int kMaxBatch = 256;

struct Geo {
    int B, L, H, H_kv, G, d, N, R;
    int la_shift, N_la;             // row j sees look-ahead keys 0..j-la_shift of N_la
    int RB, n_rb, tpr, dpad, max_splits;
    int64_t T;
    float scale;
    int64_t cu[kMaxBatch + 1];
};

__device__ __forceinline__ void load8(const __nv_bfloat16* src, float* dst) {
    uint4 v = *reinterpret_cast<const uint4*>(src);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(p[i]);
        dst[2 * i] = f.x;
        dst[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ void load8(const float* src, float* dst) {
    float4 a = reinterpret_cast<const float4*>(src)[0];
    float4 b = reinterpret_cast<const float4*>(src)[1];
    dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
    dst[4] = b.x; dst[5] = b.y; dst[6] = b.z; dst[7] = b.w;
}

__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }

__device__ __forceinline__ float dot_smem(const float* a, const float* b, int d) {
    float s = 0.f;
    for (int k = 0; k < d; k += 4) {
        float4 x = *reinterpret_cast<const float4*>(a + k);
        float4 y = *reinterpret_cast<const float4*>(b + k);
        s = fmaf(x.x, y.x, s);
        s = fmaf(x.y, y.y, s);
        s = fmaf(x.z, y.z, s);
        s = fmaf(x.w, y.w, s);
    }
    return s;
}

// Merge softmax statistics (m2, z2) into (m, z): z is a sum of exp(. - m).
__device__ __forceinline__ void merge(float& m, float& z, float m2, float z2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) { m = m2; z = z2; return; }
    float mx = fmaxf(m, m2);
    z = z * expf(m - mx) + z2 * expf(m2 - mx);
    m = mx;
}

struct Slab {
    int b, l, g, rb;
    int64_t m0, Mb;
};

__device__ __forceinline__ Slab slab_of(const Geo& geo, int y) {
    Slab s;
    int sl = y / geo.n_rb;
    s.rb = y % geo.n_rb;
    s.b = sl / (geo.L * geo.H_kv);
    s.l = (sl / geo.H_kv) % geo.L;
    s.g = sl % geo.H_kv;
    s.m0 = geo.cu[s.b];
    s.Mb = geo.cu[s.b + 1] - s.m0;
    return s;
}

template <typename In>
__device__ __forceinline__ void load_q_rows(const Geo& geo, const Slab& s, const In* Q, int r0,
                                            int nr, float* Qs) {
    const int c8n = geo.d / 8;
    for (int idx = threadIdx.x; idx < nr * c8n; idx += kThreads) {
        int rr = idx / c8n, c8 = idx % c8n;
        int r = r0 + rr, j = r / geo.G, h = s.g * geo.G + r % geo.G;
        const In* src = Q + ((((int64_t)s.b * geo.N + j) * geo.L + s.l) * geo.H + h) * geo.d + c8 * 8;
        load8(src, Qs + rr * geo.dpad + c8 * 8);
    }
}

template <typename In>
__device__ __forceinline__ void load_k_tile(const Geo& geo, const In* Kslab, int64_t ts, int nt,
                                            float* Ks) {
    const int c8n = geo.d / 8;
    for (int idx = threadIdx.x; idx < nt * c8n; idx += kThreads) {
        int t = idx / c8n, c8 = idx % c8n;
        load8(Kslab + (ts + t) * geo.d + c8 * 8, Ks + t * geo.dpad + c8 * 8);
    }
}

// (1) partial softmax statistics of every row over one split of the prompt.
template <typename In>
__global__ void __launch_bounds__(kThreads) stats_kernel(const Geo geo, const In* __restrict__ Q,
                                                         const In* __restrict__ K,
                                                         float2* __restrict__ partials) {
    extern __shared__ __align__(16) float sm[];
    const Slab s = slab_of(geo, blockIdx.y);
    const int split = blockIdx.x;
    const int64_t t_begin = (int64_t)split * kSplit;
    if (t_begin >= s.Mb) return;
    const int64_t t_end = min(t_begin + (int64_t)kSplit, s.Mb);
    const int r0 = s.rb * geo.RB, nr = min(geo.RB, geo.R - r0);
    float* Qs = sm;
    float* Ks = sm + geo.RB * geo.dpad;
    load_q_rows(geo, s, Q, r0, nr, Qs);

    const int rr = threadIdx.x / geo.tpr, tq = threadIdx.x % geo.tpr;
    const bool row_ok = rr < nr;
    const In* Kslab = K + (((int64_t)s.l * geo.H_kv + s.g) * geo.T + s.m0) * geo.d;
    float m = -INFINITY, z = 0.f;
    for (int64_t ts = t_begin; ts < t_end; ts += kSub) {
        const int nt = (int)min((int64_t)kSub, t_end - ts);
        __syncthreads();
        load_k_tile(geo, Kslab, ts, nt, Ks);
        __syncthreads();
        if (row_ok) {
            for (int t = tq; t < nt; t += geo.tpr) {
                float x = dot_smem(Qs + rr * geo.dpad, Ks + t * geo.dpad, geo.d) * geo.scale;
                if (x > m) { z = z * expf(m - x) + 1.f; m = x; }
                else       { z += expf(x - m); }
            }
        }
    }
    for (int o = geo.tpr / 2; o > 0; o >>= 1) {
        float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        float z2 = __shfl_xor_sync(0xffffffffu, z, o);
        merge(m, z, m2, z2);
    }
    if (row_ok && tq == 0) {
        int64_t sl = blockIdx.y / geo.n_rb;
        partials[(sl * geo.R + r0 + rr) * geo.max_splits + split] = make_float2(m, z);
    }
}

// (2) lse of every row: merge the split statistics in split order, then the
// causal look-ahead keys 0..j of look-ahead step j.
template <typename In>
__global__ void __launch_bounds__(kThreads) combine_kernel(const Geo geo, const In* __restrict__ Q,
                                                           const In* __restrict__ Kla,
                                                           const float2* __restrict__ partials,
                                                           float* __restrict__ lse) {
    const int sl = blockIdx.x;
    const int b = sl / (geo.L * geo.H_kv), l = (sl / geo.H_kv) % geo.L, g = sl % geo.H_kv;
    const int64_t Mb = geo.cu[b + 1] - geo.cu[b];
    const int ns = (int)((Mb + kSplit - 1) / kSplit);
    for (int r = threadIdx.x; r < geo.R; r += blockDim.x) {
        float m = -INFINITY, z = 0.f;
        for (int sp = 0; sp < ns; ++sp) {
            float2 p = partials[((int64_t)sl * geo.R + r) * geo.max_splits + sp];
            merge(m, z, p.x, p.y);
        }
        const int j = r / geo.G, h = g * geo.G + r % geo.G;
        const In* q = Q + ((((int64_t)b * geo.N + j) * geo.L + l) * geo.H + h) * geo.d;
        for (int k = 0; k <= j - geo.la_shift; ++k) {
            const In* kk = Kla + ((((int64_t)b * geo.L + l) * geo.H_kv + g) * geo.N_la + k) * geo.d;
            float u = 0.f;
            for (int t = 0; t < geo.d; ++t) u = fmaf(to_f(q[t]), to_f(kk[t]), u);
            merge(m, z, u * geo.scale, 1.f);
        }
        lse[(int64_t)sl * geo.R + r] = m + logf(z);
    }
}

// (2') lse given by the caller: lse_in[b, l, h, j] into this path's [slab, row]
// layout, row r = j*G + h % G of slab (b*L + l)*H_kv + h / G.
__global__ void lse_in_kernel(const Geo geo, const float* __restrict__ lse_in, float* __restrict__ lse) {
    const int64_t n = (int64_t)geo.B * geo.L * geo.H_kv * geo.R;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t sl = i / geo.R;
        const int r = (int)(i % geo.R);
        const int64_t bl = sl / geo.H_kv;           // b*L + l
        const int g = (int)(sl % geo.H_kv);
        const int j = r / geo.G, h = g * geo.G + r % geo.G;
        lse[i] = lse_in[(bl * geo.H + h) * geo.N + j];
    }
}

// (3) normalised weights, max over the heads of the group, atomicMax across
// KV heads and layers.  Weights are >= 0, so their IEEE bits order like
// unsigned integers.
template <typename In>
__global__ void __launch_bounds__(kThreads) normmax_kernel(const Geo geo, const In* __restrict__ Q,
                                                           const In* __restrict__ K,
                                                           const float* __restrict__ lse,
                                                           unsigned* __restrict__ acc) {
    extern __shared__ __align__(16) float sm[];
    const Slab s = slab_of(geo, blockIdx.y);
    const int64_t t_begin = (int64_t)blockIdx.x * kSplit;
    if (t_begin >= s.Mb) return;
    const int64_t t_end = min(t_begin + (int64_t)kSplit, s.Mb);
    const int r0 = s.rb * geo.RB, nr = min(geo.RB, geo.R - r0);
    float* Qs = sm;
    float* Ks = Qs + geo.RB * geo.dpad;
    float* Ys = Ks + kSub * geo.dpad;                 // [RB][kSub + 1]
    load_q_rows(geo, s, Q, r0, nr, Qs);
    const int64_t sl = blockIdx.y / geo.n_rb;
    const int rr = threadIdx.x / geo.tpr, tq = threadIdx.x % geo.tpr;
    const bool row_ok = rr < nr;
    const float my_lse = row_ok ? lse[sl * geo.R + r0 + rr] : 0.f;
    const In* Kslab = K + (((int64_t)s.l * geo.H_kv + s.g) * geo.T + s.m0) * geo.d;
    const int nj = nr / geo.G, j0 = r0 / geo.G;
    for (int64_t ts = t_begin; ts < t_end; ts += kSub) {
        const int nt = (int)min((int64_t)kSub, t_end - ts);
        __syncthreads();
        load_k_tile(geo, Kslab, ts, nt, Ks);
        __syncthreads();
        if (row_ok) {
            for (int t = tq; t < nt; t += geo.tpr) {
                float x = dot_smem(Qs + rr * geo.dpad, Ks + t * geo.dpad, geo.d) * geo.scale;
                Ys[rr * (kSub + 1) + t] = x - my_lse;
            }
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < nj * nt; idx += kThreads) {
            int jj = idx / nt, t = idx % nt;
            float v = -INFINITY;
            for (int hh = 0; hh < geo.G; ++hh) v = fmaxf(v, Ys[(jj * geo.G + hh) * (kSub + 1) + t]);
            float w = expf(v);
            atomicMax(acc + (int64_t)(j0 + jj) * geo.T + s.m0 + ts + t, __float_as_uint(w));
        }
    }
}

// (4) importance[i] = (sum_j acc[j,i]) / N, j in order.
__global__ void finalize_kernel(int N, int64_t T, const unsigned* __restrict__ acc,
                                float* __restrict__ imp) {
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < T;
         t += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int j = 0; j < N; ++j) s += __uint_as_float(acc[(int64_t)j * T + t]);
        imp[t] = s / (float)N;
    }
}

__global__ void fill_kernel(int64_t T, float v, float* __restrict__ out) {
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < T;
         t += (int64_t)gridDim.x * blockDim.x)
        out[t] = v;
}

int pow2_at_least(int x) { int p = 1; while (p < x) p <<= 1; return p; }

bool make_geo(const ScoreProblem& p, Geo& g) {
    if (p.B > kMaxBatch) return false;
    g.B = p.B; g.L = p.L; g.H = p.H; g.H_kv = p.H_kv; g.G = p.H / p.H_kv; g.d = p.d; g.N = p.N;
    g.la_shift = p.la_shift; g.N_la = p.N - p.la_shift;
    g.R = p.N * g.G;
    g.RB = std::min(g.R, (kRowsMax / g.G) * g.G);
    if (g.RB < 1) g.RB = g.G;          // G > 64: one look-ahead step per CTA
    g.n_rb = (g.R + g.RB - 1) / g.RB;
    int rp = pow2_at_least(g.RB);
    g.tpr = std::max(1, std::min(32, kThreads / rp));
    g.dpad = g.d + 4;
    g.max_splits = (int)std::max<int64_t>(1, (p.max_M + kSplit - 1) / kSplit);
    g.T = p.T;
    g.scale = 1.0f / sqrtf((float)p.d);
    for (int b = 0; b <= p.B; ++b) g.cu[b] = p.cu_M_host[b];
    return true;
}

struct Layout {
    size_t partials, lse, acc, total;
};

Layout layout_of(const ScoreProblem& p) {
    const int G = p.H / p.H_kv;
    const int64_t R = (int64_t)p.N * G, slabs = (int64_t)p.B * p.L * p.H_kv;
    const int64_t max_splits = std::max<int64_t>(1, (p.max_M + kSplit - 1) / kSplit);
    Carve c;
    Layout lo;
    lo.partials = c.take(sizeof(float2) * slabs * R * max_splits);
    lo.lse = c.take(sizeof(float) * slabs * R);
    lo.acc = c.take(sizeof(unsigned) * (size_t)p.N * p.T);
    lo.total = c.off;
    return lo;
}

template <typename In>
sp_status launch_typed(const ScoreProblem& p, const Geo& geo, const Layout& lo, char* ws,
                       cudaStream_t st) {
    const In* Q = static_cast<const In*>(p.Q);
    const In* K = static_cast<const In*>(p.K);
    const In* Kla = static_cast<const In*>(p.Kla);
    float2* partials = reinterpret_cast<float2*>(ws + lo.partials);
    float* lse = reinterpret_cast<float*>(ws + lo.lse);
    unsigned* acc = reinterpret_cast<unsigned*>(ws + lo.acc);
    const int slabs = geo.B * geo.L * geo.H_kv;

    SP_CUDA_TRY(cudaMemsetAsync(acc, 0, sizeof(unsigned) * (size_t)geo.N * geo.T, st));
    size_t sm_stats = sizeof(float) * (size_t)(geo.RB + kSub) * geo.dpad;
    size_t sm_norm = sm_stats + sizeof(float) * (size_t)geo.RB * (kSub + 1);
    SP_CUDA_TRY(cudaFuncSetAttribute(stats_kernel<In>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sm_stats));
    SP_CUDA_TRY(cudaFuncSetAttribute(normmax_kernel<In>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)sm_norm));
    dim3 grid(geo.max_splits, slabs * geo.n_rb);
    if (p.lse_mode) {
        const int64_t n = (int64_t)slabs * geo.R;
        lse_in_kernel<<<(int)std::min<int64_t>((n + 255) / 256, 1024), 256, 0, st>>>(geo, p.lse_in, lse);
        SP_LAUNCH_CHECK();
    } else {
        stats_kernel<In><<<grid, kThreads, sm_stats, st>>>(geo, Q, K, partials);
        SP_LAUNCH_CHECK();
        combine_kernel<In><<<slabs, kThreads, 0, st>>>(geo, Q, Kla, partials, lse);
        SP_LAUNCH_CHECK();
    }
    normmax_kernel<In><<<grid, kThreads, sm_norm, st>>>(geo, Q, K, lse, acc);
    SP_LAUNCH_CHECK();
    int blocks = (int)std::min<int64_t>((geo.T + 255) / 256, 4096);
    finalize_kernel<<<std::max(blocks, 1), 256, 0, st>>>(geo.N, geo.T, acc, p.importance);
    SP_LAUNCH_CHECK();
    return SP_OK;
}

}  // namespace

size_t score_simple_ws_bytes(const ScoreProblem& p) { return layout_of(p).total; }

sp_status score_simple_launch(const ScoreProblem& p, void* ws, cudaStream_t st) {
    Geo geo;
    if (!make_geo(p, geo)) {
        set_error("sp_score: batch of %d prompts exceeds the supported %d", p.B, kMaxBatch);
        return SP_EUNSUPPORTED;
    }
    SP_CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(WsHeader), st));
    if (p.T == 0) return SP_OK;
    if (p.N == 0) {
        int blocks = (int)std::min<int64_t>((p.T + 255) / 256, 4096);
        fill_kernel<<<blocks, 256, 0, st>>>(p.T, 1.0f, p.importance);
        SP_LAUNCH_CHECK();
        return SP_OK;
    }
    const Layout lo = layout_of(p);
    char* w = static_cast<char*>(ws);
    if (p.dtype == SP_BF16) return launch_typed<__nv_bfloat16>(p, geo, lo, w, st);
    return launch_typed<float>(p, geo, lo, w, st);
}

}  // namespace sp
