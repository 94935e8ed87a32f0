// Sparse-prefill input gather: the kept tokens' IDs and original position IDs,
// packed request after request for the target's prefill (paper review "Speculative
// Prefill ...", section "core algorithm: position ID recovery"; llama.cpp guide,
// "How It Works: sparse prefill").  Decoding continues at position M_b.
#include "sp_common.cuh"

namespace sp {
namespace {

constexpr int kMaxGatherBatch = 256;

struct GatherGeo {
    int B;
    int64_t cu[kMaxGatherBatch + 1];   // request offsets in token_ids / kept_pos
};

// cu_kept[b] = sum of n_kept[b'] for b' < b (one thread; B <= 256).
__global__ void kept_offsets_kernel(int B, const int64_t* __restrict__ n_kept, int64_t* __restrict__ cu_kept) {
    if (threadIdx.x == 0) {
        int64_t run = 0;
        for (int b = 0; b < B; ++b) {
            cu_kept[b] = run;
            run += n_kept[b];
        }
        cu_kept[B] = run;
    }
}

// Block (x, b): kept entries i = x*256 + t of request b.
__global__ void __launch_bounds__(256) gather_kernel(const GatherGeo geo, const int32_t* __restrict__ token_ids,
                                                     const int32_t* __restrict__ kept,
                                                     const int64_t* __restrict__ n_kept,
                                                     const int64_t* __restrict__ cu_kept,
                                                     int32_t* __restrict__ out_tokens,
                                                     int32_t* __restrict__ out_positions) {
    const int b = blockIdx.y;
    const int64_t n = n_kept[b], base = geo.cu[b], dst = cu_kept[b];
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t pos = kept[base + i];
        if (out_tokens) out_tokens[dst + i] = token_ids[base + pos];
        if (out_positions) out_positions[dst + i] = pos;
    }
}

}  // namespace

sp_status gather_launch(const int32_t* token_ids, int B, const int64_t* cu_M_host, const int32_t* kept_pos,
                        const int64_t* n_kept, int32_t* out_tokens, int32_t* out_positions, int64_t* cu_kept,
                        cudaStream_t st) {
    if (B > kMaxGatherBatch) {
        set_error("sp_gather_kept: batch of %d prompts exceeds the supported %d", B, kMaxGatherBatch);
        return SP_EUNSUPPORTED;
    }
    GatherGeo geo;
    geo.B = B;
    int64_t max_M = 0;
    for (int b = 0; b <= B; ++b) geo.cu[b] = cu_M_host[b];
    for (int b = 0; b < B; ++b) max_M = std::max<int64_t>(max_M, cu_M_host[b + 1] - cu_M_host[b]);
    kept_offsets_kernel<<<1, 32, 0, st>>>(B, n_kept, cu_kept);
    SP_LAUNCH_CHECK();
    if (max_M == 0 || B == 0) return SP_OK;
    const int bx = (int)std::min<int64_t>((max_M + 255) / 256, 1024);
    gather_kernel<<<dim3(bx, B), 256, 0, st>>>(geo, token_ids, kept_pos, n_kept, cu_kept, out_tokens,
                                                out_positions);
    SP_LAUNCH_CHECK();
    return SP_OK;
}

}  // namespace sp
