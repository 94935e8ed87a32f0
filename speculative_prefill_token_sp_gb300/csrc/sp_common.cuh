// Shared definitions of the libspecprefill CUDA sources (internal, not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/specprefill.h"

namespace sp {

// Every workspace starts with this header.  Kernels record run-time problems
// in `status` (first writer wins); sp_workspace_status reads it back.
struct WsHeader {
    int32_t status;     // sp_status, 0 = OK
    int32_t where;      // which wait / check gave up (for diagnostics)
    int32_t aux[62];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

// Bump allocator over a caller-owned workspace (offsets only, no allocation).
struct Carve {
    size_t off = sizeof(WsHeader);
    size_t take(size_t bytes) { size_t o = off; off = align_up(off + bytes); return o; }
};

__device__ __forceinline__ void record_error(WsHeader* h, int code, int where) {
    if (atomicCAS(&h->status, 0, code) == 0) h->where = where;
}

// Thread-local last-error message of the host API.
void set_error(const char* fmt, ...);
void clear_error();
const char* last_error_text();

// Problem description shared by the scoring paths.  Single prompts are a
// batch of one.  cu_M lives on the device (inside the workspace).
struct ScoreProblem {
    const void* Q;          // [B, N, L, H, d]
    const void* K;          // [L, H_kv, T, d]
    const void* Kla;        // [B, L, H_kv, N, d]; unused when lse_in is given
    const float* lse_in;    // [B, L, H, N] softmax normalisers given by the caller (lse_mode)
    bool lse_mode;          // sp_score_lse: lse_in replaces the statistics pass
    int la_shift;           // row j sees look-ahead keys 0..j-la_shift (1: row 0 is the prefill's last query);
                            // K_la holds N - la_shift keys per (layer, KV head)
    float* importance;      // [T]
    const int64_t* cu_M_host;   // [B+1] host copy
    int B, L, H, H_kv, d, N;
    int64_t T, max_M;
    sp_dtype dtype;
};

// Host launchers (defined in score_*.cu / select.cu).
size_t score_simple_ws_bytes(const ScoreProblem& p);
sp_status score_simple_launch(const ScoreProblem& p, void* ws, cudaStream_t st);

struct SelectProblem {
    const float* importance;    // [T]
    const int64_t* cu_M_host;   // [B+1]
    int B;
    int64_t T, max_M, total_chunks, max_nc;
    int chunk, pool_k;
    sp_mode mode;
    double rate;
    bool has_boost;
    sp_boost boost;
    int32_t* kept_pos;          // [T]
    int64_t* n_kept;            // [B]
    bool has_rules;             // the guide's v2 keep rules (sp_select_rules)
    sp_keep_rules rules;
};
size_t select_ws_bytes(const SelectProblem& p);
sp_status select_launch(const SelectProblem& p, void* ws, cudaStream_t st);

// Argument checks of a single-prompt selection (defined in abi.cu).  On
// success fills *out; cu_storage (2 entries) must outlive *out.
sp_status select_validate_single(const char* fn, const float* importance, int64_t M, int chunk, int pool_k,
                                 sp_mode mode, double rate, const sp_boost* boost, int32_t* kept_pos,
                                 int64_t* n_kept, SelectProblem* out, int64_t* cu_storage);

#define SP_CUDA_TRY(expr)                                                          \
    do {                                                                           \
        cudaError_t _e = (expr);                                                   \
        if (_e != cudaSuccess) {                                                   \
            ::sp::set_error("%s failed: %s (%s:%d)", #expr, cudaGetErrorString(_e), \
                            __FILE__, __LINE__);                                   \
            return SP_ECUDA;                                                       \
        }                                                                          \
    } while (0)

// Counts kernel launches (read by sp_kernel_launches).
void count_launch();

#define SP_LAUNCH_CHECK()                                                          \
    do {                                                                           \
        ::sp::count_launch();                                                      \
        cudaError_t _e = cudaGetLastError();                                       \
        if (_e != cudaSuccess) {                                                   \
            ::sp::set_error("kernel launch failed: %s (%s:%d)",                    \
                            cudaGetErrorString(_e), __FILE__, __LINE__);           \
            return SP_ECUDA;                                                       \
        }                                                                          \
    } while (0)

}  // namespace sp
