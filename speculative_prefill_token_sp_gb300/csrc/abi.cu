// extern "C" entry points of libspecprefill.so (declared in include/specprefill.h).
//
// Validation happens here, before anything is enqueued; the kernels live in
// score_*.cu and select.cu.
#include "sp_common.cuh"

#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <vector>

namespace sp {

namespace {
thread_local char g_last_error[512] = "";
}

void set_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

void clear_error() { g_last_error[0] = '\0'; }

const char* last_error_text() { return g_last_error; }

namespace {
std::atomic<uint64_t> g_launches{0};
}
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

// Implemented in gather.cu.
sp_status gather_launch(const int32_t* token_ids, int B, const int64_t* cu_M_host, const int32_t* kept_pos,
                        const int64_t* n_kept, int32_t* out_tokens, int32_t* out_positions, int64_t* cu_kept,
                        cudaStream_t st);

// Implemented in score_tc.cu: the tensor-core path for the bf16 shapes it covers.
bool score_tc_supported(const ScoreProblem& p);
size_t score_tc_ws_bytes(const ScoreProblem& p);
sp_status score_tc_launch(const ScoreProblem& p, void* ws, cudaStream_t st);
unsigned long long score_tc_set_exchange_wait_ns(unsigned long long ns);
bool score_tc_plan_of(int L, int H, int H_kv, int d, int64_t M, int N, int sms, int out[9]);

}  // namespace sp

using namespace sp;

namespace {

constexpr int kMaxBatch = 256;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sp_status check_shape(const char* fn, int L, int H, int H_kv, int d, int N, sp_dtype dtype) {
    if (L < 1 || H < 1 || H_kv < 1) {
        set_error("%s: L, H and H_kv must be >= 1 (got %d, %d, %d)", fn, L, H, H_kv);
        return SP_EINVAL;
    }
    if (H % H_kv != 0) {
        set_error("%s: H (%d) must be a multiple of H_kv (%d)", fn, H, H_kv);
        return SP_EINVAL;
    }
    if (d < 8 || d > 256 || d % 8 != 0) {
        set_error("%s: head dim d must be a multiple of 8 in [8, 256] (got %d)", fn, d);
        return d < 1 ? SP_EINVAL : SP_EUNSUPPORTED;
    }
    if (N < 0) {
        set_error("%s: N must be >= 0 (got %d)", fn, N);
        return SP_EINVAL;
    }
    if ((int64_t)N * (H / H_kv) > 256) {
        set_error("%s: N * H / H_kv = %lld exceeds 256 query rows per KV head", fn,
                  (long long)N * (H / H_kv));
        return SP_EUNSUPPORTED;
    }
    if (dtype != SP_BF16 && dtype != SP_F32) {
        set_error("%s: unknown dtype %d", fn, (int)dtype);
        return SP_EINVAL;
    }
    return SP_OK;
}

sp_status check_cu(const char* fn, int B, const int64_t* cu) {
    if (B < 1 || cu == nullptr) {
        set_error("%s: need B >= 1 and a host cu_M array of B+1 entries", fn);
        return SP_EINVAL;
    }
    if (B > kMaxBatch) {
        set_error("%s: at most %d prompts per call (got %d)", fn, kMaxBatch, B);
        return SP_EUNSUPPORTED;
    }
    if (cu[0] != 0) {
        set_error("%s: cu_M[0] must be 0 (got %lld)", fn, (long long)cu[0]);
        return SP_EINVAL;
    }
    for (int b = 0; b < B; ++b) {
        if (cu[b + 1] < cu[b]) {
            set_error("%s: cu_M must be non-decreasing (cu_M[%d]=%lld > cu_M[%d]=%lld)", fn, b,
                      (long long)cu[b], b + 1, (long long)cu[b + 1]);
            return SP_EINVAL;
        }
        if (cu[b + 1] - cu[b] > (int64_t)INT32_MAX) {
            set_error("%s: prompt %d is longer than 2^31-1 tokens", fn, b);
            return SP_EUNSUPPORTED;
        }
    }
    return SP_OK;
}

ScoreProblem make_score_problem(const void* Q, const void* K, const void* Kla, int B, const int64_t* cu,
                                int L, int H, int H_kv, int d, int N, sp_dtype dtype, float* imp) {
    ScoreProblem p;
    p.Q = Q; p.K = K; p.Kla = Kla; p.importance = imp; p.cu_M_host = cu;
    p.lse_in = nullptr;
    p.lse_mode = false;
    p.la_shift = 0;
    p.B = B; p.L = L; p.H = H; p.H_kv = H_kv; p.d = d; p.N = N; p.dtype = dtype;
    p.T = cu[B];
    p.max_M = 0;
    for (int b = 0; b < B; ++b) p.max_M = std::max<int64_t>(p.max_M, cu[b + 1] - cu[b]);
    return p;
}

size_t score_ws(const ScoreProblem& p) {
    size_t a = score_simple_ws_bytes(p);
    if (score_tc_supported(p)) a = std::max(a, score_tc_ws_bytes(p));
    return a;
}

sp_status run_score(const char* fn, const ScoreProblem& p, void* ws, size_t ws_bytes, void* stream) {
    const size_t need = score_ws(p);
    if (p.T > 0 && p.N > 0) {
        const void* third = p.lse_mode ? static_cast<const void*>(p.lse_in) : p.Kla;
        const bool third_needed = p.lse_mode || p.N > p.la_shift;     // look-ahead keys exist
        if (!p.Q || !p.K || (third_needed && !third)) {
            set_error("%s: null input pointer", fn);
            return SP_EINVAL;
        }
        if (!aligned16(p.Q) || !aligned16(p.K) || (!p.lse_mode && third_needed && !aligned16(p.Kla)) ||
            (p.lse_mode && reinterpret_cast<uintptr_t>(p.lse_in) % 4 != 0)) {
            set_error("%s: input pointers must be 16-byte aligned (lse: 4-byte)", fn);
            return SP_EINVAL;
        }
    }
    if (p.T > 0 && !p.importance) {
        set_error("%s: null importance pointer", fn);
        return SP_EINVAL;
    }
    if (!ws) {
        set_error("%s: null workspace", fn);
        return SP_EINVAL;
    }
    if (ws_bytes < need) {
        set_error("%s: workspace of %zu bytes is smaller than the %zu required", fn, ws_bytes, need);
        return SP_ENOMEM;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    sp_status s = (p.T > 0 && p.N > 0 && score_tc_supported(p)) ? score_tc_launch(p, ws, st)
                                                                : score_simple_launch(p, ws, st);
    if (s == SP_OK) clear_error();
    return s;
}

sp_status check_select_params(const char* fn, int chunk, int pool_k, sp_mode mode, double rate,
                              const sp_boost* boost) {
    if (chunk < 1) {
        set_error("%s: chunk must be >= 1 (got %d)", fn, chunk);
        return SP_EINVAL;
    }
    if (pool_k < 1 || pool_k % 2 == 0) {
        set_error("%s: pool_k must be odd and >= 1 (got %d)", fn, pool_k);
        return SP_EINVAL;
    }
    if (mode != SP_SELECT_TOPK && mode != SP_SELECT_MASS) {
        set_error("%s: unknown selection mode %d", fn, (int)mode);
        return SP_EINVAL;
    }
    if (!(rate > 0.0 && rate <= 1.0)) {
        set_error("%s: keep_rate / mass must be in (0, 1] (got %g)", fn, rate);
        return SP_EINVAL;
    }
    if (mode == SP_SELECT_MASS && pool_k != 1) {
        set_error("%s: cumulative-mass mode takes no pooling (pool_k must be 1, got %d)", fn, pool_k);
        return SP_EINVAL;
    }
    if (boost && (boost->first_n < 0 || boost->last_n < 0)) {
        set_error("%s: boost ranges must be >= 0", fn);
        return SP_EINVAL;
    }
    return SP_OK;
}

SelectProblem make_select_problem(const float* imp, int B, const int64_t* cu, int chunk, int pool_k,
                                  sp_mode mode, double rate, const sp_boost* boost, int32_t* kept,
                                  int64_t* n_kept) {
    SelectProblem p;
    p.importance = imp; p.cu_M_host = cu; p.B = B; p.T = cu[B];
    p.chunk = chunk; p.pool_k = pool_k; p.mode = mode; p.rate = rate;
    p.has_boost = boost != nullptr;
    if (boost) p.boost = *boost;
    else p.boost = sp_boost{0, 1.0, 0, 1.0, 0};
    p.kept_pos = kept; p.n_kept = n_kept;
    p.has_rules = false;
    p.rules = sp_keep_rules{0, 0, 0};
    p.max_M = 0; p.total_chunks = 0; p.max_nc = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t Mb = cu[b + 1] - cu[b];
        const int64_t nc = (Mb + chunk - 1) / chunk;
        p.max_M = std::max(p.max_M, Mb);
        p.max_nc = std::max(p.max_nc, nc);
        p.total_chunks += nc;
    }
    return p;
}

sp_status run_select(const char* fn, const SelectProblem& p, void* ws, size_t ws_bytes, void* stream) {
    if (p.T > 0 && (!p.importance || !p.kept_pos)) {
        set_error("%s: null importance or kept_pos pointer", fn);
        return SP_EINVAL;
    }
    if (!p.n_kept || !ws) {
        set_error("%s: null n_kept or workspace pointer", fn);
        return SP_EINVAL;
    }
    const size_t need = select_ws_bytes(p);
    if (ws_bytes < need) {
        set_error("%s: workspace of %zu bytes is smaller than the %zu required", fn, ws_bytes, need);
        return SP_ENOMEM;
    }
    sp_status s = select_launch(p, ws, static_cast<cudaStream_t>(stream));
    if (s == SP_OK) clear_error();
    return s;
}

}  // namespace

namespace sp {

// Validation and problem set-up of sp_select, shared with the entry point in
// select_noalloc.cu.
sp_status select_validate_single(const char* fn, const float* importance, int64_t M, int chunk, int pool_k,
                                 sp_mode mode, double rate, const sp_boost* boost, int32_t* kept_pos,
                                 int64_t* n_kept, SelectProblem* out, int64_t* cu_storage) {
    if (M < 0 || M > (int64_t)INT32_MAX) {
        set_error("%s: M must be in [0, 2^31-1] (got %lld)", fn, (long long)M);
        return M < 0 ? SP_EINVAL : SP_EUNSUPPORTED;
    }
    sp_status s = check_select_params(fn, chunk, pool_k, mode, rate, boost);
    if (s != SP_OK) return s;
    if (M > 0 && (!importance || !kept_pos)) {
        set_error("%s: null importance or kept_pos pointer", fn);
        return SP_EINVAL;
    }
    if (!n_kept) {
        set_error("%s: null n_kept pointer", fn);
        return SP_EINVAL;
    }
    cu_storage[0] = 0;
    cu_storage[1] = M;
    *out = make_select_problem(importance, 1, cu_storage, chunk, pool_k, mode, rate, boost, kept_pos, n_kept);
    return SP_OK;
}

}  // namespace sp

extern "C" {

size_t sp_score_workspace_size(int L, int H, int H_kv, int d, int64_t M, int N, sp_dtype dtype) {
    if (M < 0 || check_shape("sp_score_workspace_size", L, H, H_kv, d, N, dtype) != SP_OK) return 0;
    int64_t cu[2] = {0, M};
    return score_ws(make_score_problem(nullptr, nullptr, nullptr, 1, cu, L, H, H_kv, d, N, dtype, nullptr));
}

sp_status sp_score(const void* Q_la, const void* K_prompt, const void* K_la, int L, int H, int H_kv,
                   int d, int64_t M, int N, sp_dtype dtype, float* importance, void* ws,
                   size_t ws_bytes, void* stream) {
    sp_status s = check_shape("sp_score", L, H, H_kv, d, N, dtype);
    if (s != SP_OK) return s;
    if (M < 0 || M > (int64_t)INT32_MAX) {
        set_error("sp_score: M must be in [0, 2^31-1] (got %lld)", (long long)M);
        return M < 0 ? SP_EINVAL : SP_EUNSUPPORTED;
    }
    int64_t cu[2] = {0, M};
    ScoreProblem p = make_score_problem(Q_la, K_prompt, K_la, 1, cu, L, H, H_kv, d, N, dtype, importance);
    return run_score("sp_score", p, ws, ws_bytes, stream);
}

size_t sp_score_prefill_workspace_size(int L, int H, int H_kv, int d, int64_t M, int N, sp_dtype dtype) {
    if (M < 0 || N < 0 || check_shape("sp_score_prefill_workspace_size", L, H, H_kv, d, N + 1, dtype) != SP_OK)
        return 0;
    int64_t cu[2] = {0, M};
    ScoreProblem p = make_score_problem(nullptr, nullptr, nullptr, 1, cu, L, H, H_kv, d, N + 1, dtype, nullptr);
    p.la_shift = 1;
    return score_ws(p);
}

sp_status sp_score_prefill(const void* Q_rows, const void* K_prompt, const void* K_la, int L, int H, int H_kv,
                           int d, int64_t M, int N, sp_dtype dtype, float* importance, void* ws,
                           size_t ws_bytes, void* stream) {
    if (N < 0) {
        set_error("sp_score_prefill: N (decode steps) must be >= 0 (got %d)", N);
        return SP_EINVAL;
    }
    sp_status s = check_shape("sp_score_prefill", L, H, H_kv, d, N + 1, dtype);
    if (s != SP_OK) return s;
    if (M < 0 || M > (int64_t)INT32_MAX) {
        set_error("sp_score_prefill: M must be in [0, 2^31-1] (got %lld)", (long long)M);
        return M < 0 ? SP_EINVAL : SP_EUNSUPPORTED;
    }
    int64_t cu[2] = {0, M};
    ScoreProblem p = make_score_problem(Q_rows, K_prompt, K_la, 1, cu, L, H, H_kv, d, N + 1, dtype, importance);
    p.la_shift = 1;
    return run_score("sp_score_prefill", p, ws, ws_bytes, stream);
}

size_t sp_score_lse_workspace_size(int L, int H, int H_kv, int d, int64_t M, int N, sp_dtype dtype) {
    if (M < 0 || check_shape("sp_score_lse_workspace_size", L, H, H_kv, d, N, dtype) != SP_OK) return 0;
    int64_t cu[2] = {0, M};
    ScoreProblem p = make_score_problem(nullptr, nullptr, nullptr, 1, cu, L, H, H_kv, d, N, dtype, nullptr);
    p.lse_mode = true;                  // the plan depends only on the mode
    return score_ws(p);
}

sp_status sp_score_lse(const void* Q_la, const void* K_prompt, const float* lse, int L, int H, int H_kv,
                       int d, int64_t M, int N, sp_dtype dtype, float* importance, void* ws,
                       size_t ws_bytes, void* stream) {
    sp_status s = check_shape("sp_score_lse", L, H, H_kv, d, N, dtype);
    if (s != SP_OK) return s;
    if (M < 0 || M > (int64_t)INT32_MAX) {
        set_error("sp_score_lse: M must be in [0, 2^31-1] (got %lld)", (long long)M);
        return M < 0 ? SP_EINVAL : SP_EUNSUPPORTED;
    }
    int64_t cu[2] = {0, M};
    ScoreProblem p = make_score_problem(Q_la, K_prompt, nullptr, 1, cu, L, H, H_kv, d, N, dtype, importance);
    p.lse_in = lse;
    p.lse_mode = true;
    return run_score("sp_score_lse", p, ws, ws_bytes, stream);
}

size_t sp_score_varlen_workspace_size(int B, const int64_t* cu_M_host, int L, int H, int H_kv, int d,
                                      int N, sp_dtype dtype) {
    if (check_cu("sp_score_varlen_workspace_size", B, cu_M_host) != SP_OK) return 0;
    if (check_shape("sp_score_varlen_workspace_size", L, H, H_kv, d, N, dtype) != SP_OK) return 0;
    return score_ws(make_score_problem(nullptr, nullptr, nullptr, B, cu_M_host, L, H, H_kv, d, N, dtype,
                                       nullptr));
}

sp_status sp_score_varlen(const void* Q_la, const void* K_prompt, const void* K_la, int B,
                          const int64_t* cu_M_host, int L, int H, int H_kv, int d, int N,
                          sp_dtype dtype, float* importance, void* ws, size_t ws_bytes, void* stream) {
    sp_status s = check_cu("sp_score_varlen", B, cu_M_host);
    if (s != SP_OK) return s;
    s = check_shape("sp_score_varlen", L, H, H_kv, d, N, dtype);
    if (s != SP_OK) return s;
    ScoreProblem p = make_score_problem(Q_la, K_prompt, K_la, B, cu_M_host, L, H, H_kv, d, N, dtype,
                                        importance);
    return run_score("sp_score_varlen", p, ws, ws_bytes, stream);
}

size_t sp_score_lse_varlen_workspace_size(int B, const int64_t* cu_M_host, int L, int H, int H_kv, int d,
                                          int N, sp_dtype dtype) {
    if (check_cu("sp_score_lse_varlen_workspace_size", B, cu_M_host) != SP_OK) return 0;
    if (check_shape("sp_score_lse_varlen_workspace_size", L, H, H_kv, d, N, dtype) != SP_OK) return 0;
    ScoreProblem p = make_score_problem(nullptr, nullptr, nullptr, B, cu_M_host, L, H, H_kv, d, N, dtype,
                                        nullptr);
    p.lse_mode = true;
    return score_ws(p);
}

sp_status sp_score_lse_varlen(const void* Q_la, const void* K_prompt, const float* lse, int B,
                              const int64_t* cu_M_host, int L, int H, int H_kv, int d, int N,
                              sp_dtype dtype, float* importance, void* ws, size_t ws_bytes, void* stream) {
    sp_status s = check_cu("sp_score_lse_varlen", B, cu_M_host);
    if (s != SP_OK) return s;
    s = check_shape("sp_score_lse_varlen", L, H, H_kv, d, N, dtype);
    if (s != SP_OK) return s;
    ScoreProblem p = make_score_problem(Q_la, K_prompt, nullptr, B, cu_M_host, L, H, H_kv, d, N, dtype,
                                        importance);
    p.lse_in = lse;
    p.lse_mode = true;
    return run_score("sp_score_lse_varlen", p, ws, ws_bytes, stream);
}

sp_status sp_gather_kept(const int32_t* token_ids, int B, const int64_t* cu_M_host, const int32_t* kept_pos,
                         const int64_t* n_kept, int32_t* out_tokens, int32_t* out_positions, int64_t* cu_kept,
                         void* stream) {
    sp_status s = check_cu("sp_gather_kept", B, cu_M_host);
    if (s != SP_OK) return s;
    if (!kept_pos || !n_kept || !cu_kept || (out_tokens && !token_ids) || (!out_tokens && !out_positions)) {
        set_error("sp_gather_kept: null pointer (kept_pos, n_kept, cu_kept, and token_ids when tokens are gathered; "
                  "at least one output)");
        return SP_EINVAL;
    }
    s = gather_launch(token_ids, B, cu_M_host, kept_pos, n_kept, out_tokens, out_positions, cu_kept,
                      static_cast<cudaStream_t>(stream));
    if (s == SP_OK) clear_error();
    return s;
}

size_t sp_select_workspace_size(int64_t M, int chunk) {
    if (M < 0 || chunk < 1) return 0;
    int64_t cu[2] = {0, M};
    return select_ws_bytes(make_select_problem(nullptr, 1, cu, chunk, 1, SP_SELECT_TOPK, 1.0, nullptr,
                                               nullptr, nullptr));
}

sp_status sp_select(const float* importance, int64_t M, int chunk, int pool_k, sp_mode mode, double rate,
                    const sp_boost* boost, int32_t* kept_pos, int64_t* n_kept, void* ws, size_t ws_bytes,
                    void* stream) {
    if (M < 0 || M > (int64_t)INT32_MAX) {
        set_error("sp_select: M must be in [0, 2^31-1] (got %lld)", (long long)M);
        return M < 0 ? SP_EINVAL : SP_EUNSUPPORTED;
    }
    sp_status s = check_select_params("sp_select", chunk, pool_k, mode, rate, boost);
    if (s != SP_OK) return s;
    int64_t cu[2] = {0, M};
    SelectProblem p = make_select_problem(importance, 1, cu, chunk, pool_k, mode, rate, boost, kept_pos,
                                          n_kept);
    return run_select("sp_select", p, ws, ws_bytes, stream);
}

size_t sp_select_rules_workspace_size(int64_t M, int chunk) {
    if (M < 0 || chunk < 1) return 0;
    int64_t cu[2] = {0, M};
    SelectProblem p = make_select_problem(nullptr, 1, cu, chunk, 1, SP_SELECT_TOPK, 1.0, nullptr, nullptr, nullptr);
    p.has_rules = true;
    return select_ws_bytes(p);
}

sp_status sp_select_rules(const float* importance, int64_t M, int chunk, int pool_k, sp_mode mode, double rate,
                          const sp_boost* boost, const sp_keep_rules* rules, int32_t* kept_pos, int64_t* n_kept,
                          void* ws, size_t ws_bytes, void* stream) {
    if (M < 0 || M > (int64_t)INT32_MAX) {
        set_error("sp_select_rules: M must be in [0, 2^31-1] (got %lld)", (long long)M);
        return M < 0 ? SP_EINVAL : SP_EUNSUPPORTED;
    }
    sp_status s = check_select_params("sp_select_rules", chunk, pool_k, mode, rate, boost);
    if (s != SP_OK) return s;
    if (rules && (rules->min_tok < 0 || rules->max_keep < 0)) {
        set_error("sp_select_rules: min_tok and max_keep must be >= 0");
        return SP_EINVAL;
    }
    if (rules && rules->min_tok > 4096) {
        set_error("sp_select_rules: min_tok is at most 4096 (got %d)", rules->min_tok);
        return SP_EUNSUPPORTED;
    }
    int64_t cu[2] = {0, M};
    SelectProblem p = make_select_problem(importance, 1, cu, chunk, pool_k, mode, rate, boost, kept_pos, n_kept);
    if (rules) {
        p.has_rules = true;
        p.rules = *rules;
    }
    return run_select("sp_select_rules", p, ws, ws_bytes, stream);
}

size_t sp_select_varlen_workspace_size(int B, const int64_t* cu_M_host, int chunk) {
    if (chunk < 1 || check_cu("sp_select_varlen_workspace_size", B, cu_M_host) != SP_OK) return 0;
    return select_ws_bytes(make_select_problem(nullptr, B, cu_M_host, chunk, 1, SP_SELECT_TOPK, 1.0,
                                               nullptr, nullptr, nullptr));
}

sp_status sp_select_varlen(const float* importance, int B, const int64_t* cu_M_host, int chunk, int pool_k,
                           sp_mode mode, double rate, const sp_boost* boost, int32_t* kept_pos,
                           int64_t* n_kept, void* ws, size_t ws_bytes, void* stream) {
    sp_status s = check_cu("sp_select_varlen", B, cu_M_host);
    if (s != SP_OK) return s;
    s = check_select_params("sp_select_varlen", chunk, pool_k, mode, rate, boost);
    if (s != SP_OK) return s;
    SelectProblem p = make_select_problem(importance, B, cu_M_host, chunk, pool_k, mode, rate, boost,
                                          kept_pos, n_kept);
    return run_select("sp_select_varlen", p, ws, ws_bytes, stream);
}

sp_status sp_workspace_status(const void* ws, void* stream) {
    if (!ws) {
        set_error("sp_workspace_status: null workspace");
        return SP_EINVAL;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WsHeader h;
    cudaError_t e = cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        set_error("sp_workspace_status: %s", cudaGetErrorString(e));
        return SP_ECUDA;
    }
    if (h.status != SP_OK) {
        set_error("device-side status %d recorded at check %d", h.status, h.where);
        return (sp_status)h.status;
    }
    return SP_OK;
}

const char* sp_last_error(void) { return last_error_text(); }

const char* sp_status_string(sp_status s) {
    switch (s) {
        case SP_OK: return "SP_OK";
        case SP_EINVAL: return "SP_EINVAL";
        case SP_ENOMEM: return "SP_ENOMEM";
        case SP_ECUDA: return "SP_ECUDA";
        case SP_EDEVICE: return "SP_EDEVICE";
        case SP_ETIMEOUT: return "SP_ETIMEOUT";
        case SP_EUNSUPPORTED: return "SP_EUNSUPPORTED";
    }
    return "SP_UNKNOWN";
}

int sp_version(void) { return 100; }

uint64_t sp_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

uint64_t sp_test_set_exchange_wait_ns(uint64_t ns) { return score_tc_set_exchange_wait_ns(ns); }

int sp_test_score_plan(int L, int H, int H_kv, int d, int64_t M, int N, int sms, int* out9) {
    if (out9 == nullptr || sms < 1 || M < 1 || N < 1) return 0;
    return score_tc_plan_of(L, H, H_kv, d, M, N, sms, out9) ? 1 : 0;
}

}  // extern "C"
