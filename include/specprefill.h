/*
 * specprefill.h -- C ABI of libspecprefill.so: SpecPrefill token-importance
 * scoring and chunk selection on one NVIDIA GB300 (sm_103a).
 *
 * The method (paper review "Speculative Prefill: Turbocharging TTFT with
 * Lightweight and Training-Free Token Importance Estimation", sections "core
 * algorithm" and "core formulas"; llama.cpp guide "SpecPrefill --
 * Implementation Guide", sections "How It Works", "v3 Improvements" and
 * "v3.1 Optimizations"): a small speculator model has a post-RoPE key cache for
 * an M-token prompt and the queries of N look-ahead decode steps.  Every
 * prompt token i gets the importance
 *
 *     importance_i = (1/N) sum_j max_{l,h} softmax(Q_{M+j,l,h} K_{l,g(h)}^T / sqrt(d))_i
 *
 * where the softmax of look-ahead step j runs over the M prompt keys and the
 * look-ahead keys 0..j.  The prompt is then cut into contiguous chunks, chunk
 * scores are averaged (and pooled), chunks are selected, and the original
 * position IDs of the kept tokens are returned in ascending order.  Decoding
 * continues at positions M, M+1, ... (paper review, "position ID recovery").
 *
 * Conventions of every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, except
 *    arguments whose name ends in "_host".  Layouts are row-major, last index
 *    contiguous.  Data pointers must be 16-byte aligned.
 *  - The library never allocates, frees or synchronises (except
 *    sp_workspace_status).  Work is enqueued on `stream` (a cudaStream_t;
 *    NULL = the legacy default stream) and runs asynchronously; outputs are
 *    valid once the stream reaches that point.
 *  - `ws` is a caller-owned device workspace of at least the size the matching
 *    *_workspace_size function returns; its contents need not be initialised
 *    and are overwritten.  One workspace must not be used by two calls that
 *    may run at the same time.
 *  - Errors: arguments are validated before anything is enqueued; on failure
 *    the call returns a non-zero sp_status, enqueues nothing and
 *    sp_last_error() describes the problem.  CUDA launch failures return
 *    SP_ECUDA.  A kernel that detects a problem at run time (a bounded wait
 *    that gave up) records it in the workspace; sp_workspace_status() reads it.
 *    Nothing aborts the process.
 */
#ifndef SPECPREFILL_H
#define SPECPREFILL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SP_OK = 0,
    SP_EINVAL = 1,        /* bad argument (shape, pointer, parameter range)          */
    SP_ENOMEM = 2,        /* workspace smaller than *_workspace_size() asks for      */
    SP_ECUDA = 3,         /* a CUDA runtime call or kernel launch failed             */
    SP_EDEVICE = 4,       /* a kernel recorded an internal error in the workspace    */
    SP_ETIMEOUT = 5,      /* a bounded device-side wait gave up                      */
    SP_EUNSUPPORTED = 6   /* valid, but outside what this build implements          */
} sp_status;

typedef enum { SP_BF16 = 0, SP_F32 = 1 } sp_dtype;

typedef enum {
    SP_SELECT_TOPK = 0,   /* chunk mean -> 1D average pool -> exactly kc chunks      */
    SP_SELECT_MASS = 1    /* v3: chunks by mean until the cumulative mass >= tau    */
} sp_mode;

/* v3 structural boost (llama.cpp guide, "v3 Improvements: Structural Token
 * Boosting" and "v3.1: Score Normalization").  Token scores are first min-max
 * normalised to [0,1] over the prompt if `normalize` != 0 (all 1.0 when every
 * score is equal), then multiplied by first_mult at positions [0, first_n) and
 * by last_mult at positions [M - last_n, M) (both when the ranges overlap).
 * The guide's defaults are {64, 1.5, 128, 1.3, 1}. */
typedef struct {
    int32_t first_n;
    double  first_mult;
    int32_t last_n;
    double  last_mult;
    int32_t normalize;
} sp_boost;

/* The guide's v2 keep rules applied after the chunk selection (llama.cpp
 * guide, "Full Source Code": select_chunks and its main program's sparse-
 * prefill cap).  min_tok > 0 sets eff_min = min(min_tok, max(4, M / 10)): a
 * prompt of at most eff_min tokens keeps every token, otherwise tokens of the
 * chunks the selection left out are added, chunk by chunk and token by token
 * in order, until eff_min are kept.  always_keep != 0 adds tokens 0, 1, 2, 3
 * and, if M > 4, M-2 and M-1.  max_keep > 0 caps the result: with n > max_keep
 * kept, every (n / max_keep)-th token is kept, at most max_keep, the last one
 * replaced by the last kept token.  The guide runs with {128, 1, 2000}. */
typedef struct {
    int32_t min_tok;        /* 0 = off; at most 4096 */
    int32_t always_keep;
    int64_t max_keep;       /* 0 = no cap */
} sp_keep_rules;

/* ------------------------------------------------------------------------ */
/* Scoring                                                                  */
/* ------------------------------------------------------------------------ */

/* Workspace bytes sp_score needs for this shape (0 if the shape is invalid). */
size_t sp_score_workspace_size(int L, int H, int H_kv, int d, int64_t M, int N, sp_dtype dtype);

/* Token importance of one prompt.
 *
 * Defines: a[l,h,j,i] = softmax over {prompt keys 0..M-1, look-ahead keys
 * 0..j} of Q_la[j,l,h,:] . key / sqrt(d), evaluated at prompt key i;
 * importance[i] = (1/N) sum_j max_{l,h} a[l,h,j,i]   (paper review, "core
 * formulas": attention score and importance aggregation; llama.cpp guide,
 * "Token Importance": max over heads, max over layers, mean over look-ahead
 * steps).  Query head h reads KV head h / (H / H_kv).
 *
 *   Q_la      [N, L, H, d]      look-ahead queries (post-RoPE), dtype
 *   K_prompt  [L, H_kv, M, d]   prompt keys (post-RoPE), dtype
 *   K_la      [L, H_kv, N, d]   look-ahead keys (post-RoPE), dtype
 *   importance[M]               fp32 output
 *   dtype     SP_BF16 or SP_F32 (all three inputs)
 *
 * Requirements: L, H, H_kv >= 1, H % H_kv == 0, 1 <= d <= 256, d % 8 == 0,
 * M >= 0, 0 <= N, N * (H / H_kv) <= 256.  N == 0 writes importance 1.0 to
 * every token (the guide's fallback when no look-ahead step was captured).
 * M == 0 is a no-op.  Accuracy: importance within 1e-3 absolute and 1e-2
 * relative of an fp64 evaluation on the same bf16 inputs; 1e-5 for fp32. */
sp_status sp_score(const void* Q_la, const void* K_prompt, const void* K_la,
                   int L, int H, int H_kv, int d, int64_t M, int N, sp_dtype dtype,
                   float* importance, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes sp_score_prefill needs (N = decode steps; 0 if the shape is invalid). */
size_t sp_score_prefill_workspace_size(int L, int H, int H_kv, int d, int64_t M, int N, sp_dtype dtype);

/* sp_score for the capture the llama.cpp guide makes ("How It Works": the
 * prefill's last row, then the look-ahead decode steps): N + 1 query rows,
 * where row 0 is the prompt's last query at prefill -- its softmax covers only
 * the M prompt keys -- and row j >= 1 is decode step j - 1, whose softmax also
 * covers look-ahead keys 0..j-1.  importance[i] = (1/(N+1)) sum_j max_{l,h} a[l,h,j,i].
 *
 *   Q_rows    [N + 1, L, H, d]  row 0: the prompt's last query; rows 1..N: decode queries
 *   K_prompt  [L, H_kv, M, d]
 *   K_la      [L, H_kv, N, d]   the decode steps' keys (may be NULL when N == 0)
 *
 * Requirements as sp_score with N + 1 rows ((N + 1) * (H / H_kv) <= 256). */
sp_status sp_score_prefill(const void* Q_rows, const void* K_prompt, const void* K_la,
                           int L, int H, int H_kv, int d, int64_t M, int N, sp_dtype dtype,
                           float* importance, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes sp_score_lse needs for this shape (0 if the shape is invalid). */
size_t sp_score_lse_workspace_size(int L, int H, int H_kv, int d, int64_t M, int N, sp_dtype dtype);

/* Token importance of one prompt when each row's softmax normaliser is
 * already known (single pass: K is read once, no statistics pass).
 *
 * Defines: importance[i] = (1/N) sum_j max_{l,h} exp(Q_la[j,l,h,:] . K[l,g,i,:] / sqrt(d)
 * - lse[l,h,j]), g = h / (H / H_kv) -- the aggregation of sp_score (paper
 * review, "core formulas"; llama.cpp guide, "Token Importance"), with lse
 * supplied by the caller.  With lse[l,h,j] the log of the sum of exp over
 * the M prompt logits and the look-ahead logits 0..j -- the normaliser the
 * speculator's own look-ahead decode attention computes -- the result equals
 * sp_score's.  The pages have no separate call for this; it is the
 * "lse-in" variant of the same definition.
 *
 *   Q_la      [N, L, H, d]      look-ahead queries (post-RoPE), dtype
 *   K_prompt  [L, H_kv, M, d]   prompt keys (post-RoPE), dtype
 *   lse       [L, H, N]         fp32 natural-log normalisers (device memory, 4-byte aligned)
 *   importance[M]               fp32 output
 *
 * Requirements and errors as sp_score; N == 0 writes 1.0 and reads no lse.
 * Accuracy: within 1e-3 absolute and 1e-2 relative of an fp64 evaluation on
 * the same inputs (bf16), 1e-5 (fp32). */
sp_status sp_score_lse(const void* Q_la, const void* K_prompt, const float* lse,
                       int L, int H, int H_kv, int d, int64_t M, int N, sp_dtype dtype,
                       float* importance, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for sp_score_varlen (cu_M_host: B+1 host prefix sums).  The
 * batch is planned for the current device's SM count: query the size with the
 * device that will run the call current (a smaller workspace is rejected with
 * SP_EINVAL, never overrun). */
size_t sp_score_varlen_workspace_size(int B, const int64_t* cu_M_host, int L, int H, int H_kv,
                                      int d, int N, sp_dtype dtype);

/* Token importance of B independent prompts in one call.  Prompt b has
 * M_b = cu_M_host[b+1] - cu_M_host[b] tokens (cu_M_host[0] == 0, non-
 * decreasing; empty prompts allowed).  Keys are packed along the token axis:
 *
 *   Q_la      [B, N, L, H, d]
 *   K_prompt  [L, H_kv, T, d]   T = cu_M_host[B]; prompt b occupies rows cu_M[b]..cu_M[b+1]-1
 *   K_la      [B, L, H_kv, N, d]
 *   importance[T]               fp32; entries of prompt b at offsets cu_M[b]..
 *
 * Same definition and requirements as sp_score, per prompt. */
sp_status sp_score_varlen(const void* Q_la, const void* K_prompt, const void* K_la,
                          int B, const int64_t* cu_M_host,
                          int L, int H, int H_kv, int d, int N, sp_dtype dtype,
                          float* importance, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for sp_score_lse_varlen (planned for the current device, as
 * sp_score_varlen_workspace_size; 0 if the shape or cu_M_host is invalid). */
size_t sp_score_lse_varlen_workspace_size(int B, const int64_t* cu_M_host, int L, int H, int H_kv,
                                          int d, int N, sp_dtype dtype);

/* sp_score_lse for B independent prompts in one call: the packing of
 * sp_score_varlen, with each prompt's row normalisers given instead of its
 * look-ahead keys (single pass per prompt, K read once).
 *
 *   Q_la      [B, N, L, H, d]
 *   K_prompt  [L, H_kv, T, d]   T = cu_M_host[B]; prompt b occupies rows cu_M[b]..cu_M[b+1]-1
 *   lse       [B, L, H, N]      fp32 natural-log normalisers of prompt b's rows (device, 4-byte aligned)
 *   importance[T]               fp32; entries of prompt b at offsets cu_M[b]..
 *
 * Same definition as sp_score_lse per prompt; requirements and errors as
 * sp_score_varlen.  lse holds all B prompts' rows; those of empty prompts are
 * not used. */
sp_status sp_score_lse_varlen(const void* Q_la, const void* K_prompt, const float* lse,
                              int B, const int64_t* cu_M_host,
                              int L, int H, int H_kv, int d, int N, sp_dtype dtype,
                              float* importance, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Selection                                                                */
/* ------------------------------------------------------------------------ */

/* Workspace bytes sp_select needs for a prompt of M tokens and this chunk size. */
size_t sp_select_workspace_size(int64_t M, int chunk);

/* Kept original position IDs of one prompt.
 *
 * Token scores x_i are the fp32 importance values as fp64, optionally
 * normalised and boosted (`boost`, NULL = neither).  Chunks are the contiguous
 * ranges [c*chunk, min((c+1)*chunk, M)), nc = ceil(M/chunk); a chunk's mean is
 * its fp64 sum (added left to right) divided by its real size (paper review,
 * chunk formula; llama.cpp guide, select_chunks).
 *
 * SP_SELECT_TOPK (rate = keep_rate, 0 < rate <= 1): chunk means are smoothed
 * by a stride-1, centred average pool of pool_k chunks (odd; an edge window
 * averages only its in-range chunks), and exactly kc = max(1,
 * ceil(f32(nc) * f32(rate))) chunks with the largest pooled score are kept,
 * ties to the lower chunk index (paper review, "chunk selection and pooling
 * denoising"; the guide's kc formula).
 *
 * SP_SELECT_MASS (rate = tau, 0 < tau <= 1; pool_k must be 1): chunks are
 * ranked by mean (descending, ties to the lower index) and the shortest ranked
 * prefix whose running sum of chunk sums (added in ranked order) reaches
 * tau * total (chunk sums added in chunk order) is kept; all chunks if it never
 * does (llama.cpp guide, "v3 Improvements: Cumulative Attention Mass
 * Selection").  Supports nc <= 16384.
 *
 *   importance [M] fp32 (finite values)
 *   kept_pos   [M] int32 output capacity; the first *n_kept entries receive the
 *              kept tokens' original positions, ascending
 *   n_kept     device int64 output
 *
 * Every fp64 operation follows the fixed order above, so the result is
 * reproducible bit for bit by any IEEE-754 implementation of the same steps. */
sp_status sp_select(const float* importance, int64_t M, int chunk, int pool_k, sp_mode mode,
                    double rate, const sp_boost* boost, int32_t* kept_pos, int64_t* n_kept,
                    void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for sp_select_rules. */
size_t sp_select_rules_workspace_size(int64_t M, int chunk);

/* sp_select followed by the keep rules (sp_keep_rules) on the same prompt.
 * kept_pos receives the final ascending positions (capacity M) and n_kept
 * their count.  rules == NULL behaves as sp_select.  Errors: SP_EINVAL for a
 * negative min_tok or max_keep, SP_EUNSUPPORTED for min_tok > 4096. */
sp_status sp_select_rules(const float* importance, int64_t M, int chunk, int pool_k, sp_mode mode,
                          double rate, const sp_boost* boost, const sp_keep_rules* rules,
                          int32_t* kept_pos, int64_t* n_kept, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for sp_select_varlen. */
size_t sp_select_varlen_workspace_size(int B, const int64_t* cu_M_host, int chunk);

/* Per-prompt selection of B packed prompts (importance packed as in
 * sp_score_varlen).  Prompt b's kept positions (relative to its own start,
 * i.e. its original position IDs) go to kept_pos[cu_M[b] ...] and its count
 * to n_kept[b] (device int64[B]).  Same rules as sp_select per prompt. */
sp_status sp_select_varlen(const float* importance, int B, const int64_t* cu_M_host, int chunk,
                           int pool_k, sp_mode mode, double rate, const sp_boost* boost,
                           int32_t* kept_pos, int64_t* n_kept, void* ws, size_t ws_bytes,
                           void* stream);

/* sp_select for callers that cannot allocate device memory.  The method's
 * pages have no counterpart to this entry point; it exists for deployment.
 *
 * Who needs it: code that runs inside a device-memory allocator or its
 * out-of-memory handler (allocating there would re-enter the allocator),
 * serving loops whose latency budget forbids cudaMalloc (it can synchronise
 * the whole device), and plug-ins that a host framework hands only input and
 * output buffers.  The caller passes inputs and outputs exactly as for
 * sp_select; the scratch lives in a fixed 3 MiB array of device memory inside
 * the library.  The array comes into being on a device when the library's
 * code is loaded there: with CUDA's lazy module loading (the default) that is
 * the first call of this entry point on the device, which looks up the
 * array's address with that device current and may itself allocate device
 * memory (the array and the selection kernels' code).  So make one call on
 * every device ahead of time -- before the allocator or out-of-memory path
 * that needs it, and before any stream capture.  Later calls allocate and
 * free nothing; the array stays until the process exits.
 *
 * Limits: one prompt, at most 65536 chunks (ceil(M / chunk)); larger requests
 * return SP_EUNSUPPORTED before any work is enqueued.  All calls on a device
 * share the array and leave their contents behind: calls whose work may
 * overlap on the GPU (e.g. on two unordered streams) race and must not be
 * issued.  Results are identical to sp_select's. */
sp_status sp_select_noalloc(const float* importance, int64_t M, int chunk, int pool_k, sp_mode mode,
                            double rate, const sp_boost* boost, int32_t* kept_pos, int64_t* n_kept,
                            void* stream);

/* ------------------------------------------------------------------------ */
/* Sparse-prefill input                                                     */
/* ------------------------------------------------------------------------ */

/* The target's sparse-prefill batch: for B packed prompts, each prompt's kept
 * token IDs and original position IDs, packed prompt after prompt (paper
 * review, "core algorithm: position ID recovery": the kept tokens keep their
 * positions and decoding continues at M_b, M_b + 1, ...).
 *
 *   token_ids     [T] int32, packed by cu_M_host (needed only if out_tokens is given)
 *   kept_pos      [T] int32, prompt b's ascending kept positions (relative to its
 *                 start) at kept_pos[cu_M[b] ...], as sp_select_varlen writes them
 *   n_kept        device int64[B], as sp_select_varlen writes it
 *   out_tokens    [T] int32 capacity or NULL: out_tokens[cu_kept[b] + i] = token_ids[cu_M[b] + kept_pos[cu_M[b] + i]]
 *   out_positions [T] int32 capacity or NULL: out_positions[cu_kept[b] + i] = kept_pos[cu_M[b] + i]
 *   cu_kept       device int64[B + 1]: prefix sums of n_kept
 *
 * Requirements: 1 <= B <= 256, cu_M_host as for sp_select_varlen; at least one
 * of out_tokens / out_positions.  No workspace. */
sp_status sp_gather_kept(const int32_t* token_ids, int B, const int64_t* cu_M_host, const int32_t* kept_pos,
                         const int64_t* n_kept, int32_t* out_tokens, int32_t* out_positions, int64_t* cu_kept,
                         void* stream);

/* ------------------------------------------------------------------------ */
/* Status                                                                   */
/* ------------------------------------------------------------------------ */

/* Synchronises `stream` and returns the run-time status a kernel recorded in
 * the workspace `ws` of the last call that used it: SP_OK, SP_ETIMEOUT (a
 * bounded wait gave up) or SP_EDEVICE.  Also returns SP_ECUDA if the stream
 * reports an error. */
sp_status sp_workspace_status(const void* ws, void* stream);

/* Message of the last failing call on this host thread ("" if none). */
const char* sp_last_error(void);

/* Name of a status code. */
const char* sp_status_string(sp_status s);

/* ABI version (major * 100 + minor). */
int sp_version(void);

/* Number of CUDA kernels this process has launched through the library
 * (all entry points, all threads).  For accounting in benchmarks. */
uint64_t sp_kernel_launches(void);

/* ------------------------------------------------------------------------ */
/* Test hook (not for production use)                                       */
/* ------------------------------------------------------------------------ */

/* Sets the limit, in nanoseconds, of the tensor-core scoring kernel's waits
 * on other CTAs' exchange entries (each token range's softmax statistics and
 * each row's lse); 0 restores the default of 4 s.  Returns the previous limit.
 * Calls enqueued afterwards use the new limit (it is read when a call is
 * planned); waits inside one CTA and the drain of its in-flight copies and
 * MMAs keep 4 s.  Tests lower it to about a microsecond so that an exchange
 * wait runs out: the kernel then records SP_ETIMEOUT in the workspace, stops
 * every warp role, waits for its in-flight copies and MMAs, frees its tensor
 * memory and returns, and sp_workspace_status reports SP_ETIMEOUT.  Process-
 * wide, not synchronised with calls running on other threads. */
uint64_t sp_test_set_exchange_wait_ns(uint64_t ns);

/* Test hook (host only, no device work): the tensor-core scoring path's plan
 * for one bf16 prompt of M tokens (L layers, H query heads, H_kv KV heads, head
 * dim d, N look-ahead steps; the first pass when N needs several) on `sms` SMs.
 * Writes nine ints to out9 (caller-owned host memory): slab classes F, CTAs per
 * class Pc, CTAs P = F * Pc, tiles of 128 tokens per CTA per slab, tiles per
 * epilogue group, landing tiles per group, held slabs per group, the
 * statistics-to-normalise lag in slabs, and the shared memory per CTA in bytes.
 * Returns 1, or 0 when that path does not take the shape (or an argument is
 * out of range); nothing is launched and nothing else is written. */
int sp_test_score_plan(int L, int H, int H_kv, int d, int64_t M, int N, int sms, int* out9);

#ifdef __cplusplus
}
#endif

#endif /* SPECPREFILL_H */
