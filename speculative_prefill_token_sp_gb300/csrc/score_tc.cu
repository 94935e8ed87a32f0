// Look-ahead attention importance on GB300 tensor cores: tcgen05.mma + TMA + TMEM.
//
// Method (paper review "Speculative Prefill ...", core formulas; llama.cpp
// guide "SpecPrefill -- Implementation Guide", Token Importance):
//   s[l,h,j,i]    = Q_la[j,l,h] . K[l,g,i] / sqrt(d)
//   lse[l,h,j]    = log(sum_i exp(s) + sum_{k<=j} exp(u_k))    (causal look-ahead keys u)
//   importance[i] = (1/N) sum_j max_{l,h} exp(s[l,h,j,i] - lse[l,h,j])
// computed as (1/N) sum_j exp(max_{l,h}(s - lse)) (exp is increasing).
//
// Design (one persistent CTA per SM, cooperative launch so that all CTAs are
// resident).  The slabs ((layer, KV head) pairs) are dealt to F classes; the
// CTAs of a class each own one fixed range of prompt tokens (multiples of 32)
// in every slab of the class, so a token's max over the class's heads and
// layers stays inside one CTA, and the F CTAs of a range combine their maxima
// once at the end (order-preserving atomicMax; with F = 1 importance is
// written directly).  A row's weights can only be normalised once its lse over
// all M tokens -- i.e. over every CTA of the class -- is known, so each slab
// has a statistics pass (P1) and, `lag` slabs later, a normalise pass (P2).
// K is read from HBM exactly once; the logits wait for P2 in TMEM.  A batch of
// prompts runs in waves: each prompt of a wave gets its own CTAs, plan and
// workspace slice in one launch (tc_score_batch_kernel).  Warp roles:
//  * warp 0 (TMA): streams the CTA's K rows (one 128-row x 128-byte box per 64
//    columns of a full tile, 32-row boxes for a slab's ragged last tile, 128B
//    swizzle) through a ring of shared-memory stages in plain order (slab after
//    slab, so every CTA reads one sequential stream), and each slab's query rows
//    (a pre-swizzled image built by tc_prep_kernel) with one bulk copy;
//  * warp 1 (MMA): tcgen05.mma, M = 128 tokens, N = 32 query rows (N*G padded),
//    K = 16 per instruction, bf16 in, fp32 accumulate into a small "landing"
//    ring of TMEM tiles per epilogue group; the CTA's k-th tile goes to group
//    k % 2, so both groups work on every slab;
//  * warps 2-17 (epilogue, two groups of eight warps; one TMEM lane = one token
//    per thread).  Each warp owns one TMEM lane quadrant (32 tokens of every
//    tile) and one half of the query rows, and works on it alone: its hand-offs
//    are mbarriers that count the warps taking part, never a barrier with
//    another warp.  P1 reads its part of a landing tile, frees it at once,
//    adds each row's exp(s - c) over its 32 tokens to the row's running sum
//    (shuffle butterflies, no shared memory), c being a per-row reference the
//    warp keeps for the slab, and stores the part again in the group's "held"
//    TMEM region as fp16 offsets s - c (half the columns, so many more slabs
//    fit).  P2 reads the held part, subtracts lse,
//    takes the max over the G heads of each look-ahead step and folds it into a
//    per-token running max in shared memory.  Held slabs never block the MMA
//    warp, so the HBM stream does not wait for the lse exchange;
//  * warp 18 (publish): merges the eight parts' statistics of each slab and
//    writes them to global memory (single 64-bit stores; a published entry
//    always has z >= 1, so a zeroed entry means "not there yet" and no fence is
//    needed);
//  * warps 19-22 (merge): a slab is merged by the CTA of its class whose range
//    index is the slab's position in the class modulo the CTAs per class: it
//    reads every CTA's entry (re-reading those still 0), adds the look-ahead
//    keys and publishes lse as (value, tag) 64-bit entries;
//  * warp 23 (fetch): waits until a slab's lse entries are all tagged and copies
//    them into a shared-memory ring for the epilogue.
// The TMA and MMA warps issue from one lane each on SM sub-partitions shared
// with busy epilogue warps, so their per-tile instruction streams are kept
// short: inline barrier waits, ring counters instead of divisions, MMA
// descriptors advanced by constants.  Epilogue warps wait with every lane and a
// vote, so the common path has no divergent branch.
//
// Units: every logit, statistic, lse and running max inside this kernel is in
// base 2 (the natural-log value times log2 e), so each weight is one exp2; the
// given lse of the lse-in variant is converted on entry and importance is
// written as exp2 of the running maxima.
//
// Precision: P1 statistics use the fp32 logits.  P2 reads w = s - c in fp16,
// c = the largest logit of the row seen so far in the slab by the warp (taken
// again whenever a value exceeds it by more than kRefMargin), so w <= 2.08 in
// natural-log units, and its rounding error is at most |w| * 2^-11 (fp16 unit
// roundoff; the same bound in either base).  A weight exp(w + c - lse) is then
// off by at most |w| * 2^-11 relative: < 1.1e-3 for 0 < w <= 2.08, < 1% for
// -20 < w <= 0, and for w <= 0 by < 1.8e-4 absolute (c <= lse, and
// exp(w) * |w| * 2^-11 peaks at w = -1).
//
// Every wait is bounded: on timeout the kernel records SP_ETIMEOUT in the
// workspace header, all roles stop, in-flight copies and MMAs are waited for
// (again bounded) and TMEM is freed before the CTA exits.
#include "sp_common.cuh"

#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>
#include <vector>
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>
#include <mutex>

namespace sp {
namespace {

constexpr int kThreads = 768;        // 24 warps
constexpr int kPubWarp = 18;         // warps 2-17: epilogue
constexpr int kMergeBase = 608;      // warps 19-22: merge
constexpr int kFetchWarp = 23;
constexpr int kEpiWarpsPerGroup = 8;
constexpr int kTileRows = 128;       // tokens per MMA tile (MMA M)
constexpr int kBoxRows = 32;         // rows per TMA box of a slab's ragged last tile (full tiles: one box)
constexpr int kUnit = 32;            // token-range granularity
constexpr int kRP = 32;              // query rows per slab, padded (MMA N)
constexpr int kMaxCtas = 256;
constexpr int kMaxTiles = 8;         // tiles per CTA per slab for slab classes and batch waves
// Tiles per CTA per slab that a plan may have at most: prompts longer than
// kMaxTiles tiles on every CTA (about 155K tokens at 152 CTAs) keep the
// tensor-core path with fewer held slabs (down to none: P2 right after P1),
// as far as the running maxima leave shared memory for two K stages (about
// 270K tokens at the 8B shape, 310K at d = 64)
constexpr int kMaxTilesLong = 16;
// How far (base-2 units) a logit may rise above its row's reference before the
// epilogue retakes the reference (3 = 2.08 in natural-log units): fp16 offsets
// below it keep the dominant values of a row to about 2^-11 relative.
constexpr float kRefMargin = 3.0f;
constexpr int kRefBytes = 16 * 16 * 4;  // 16 row references per epilogue warp
constexpr int kMaxHeld = 12;         // held slabs per epilogue group
constexpr int kRing = 16;            // entries of the lse ring
constexpr int kStatsRing = 4;        // entries of the statistics ring
constexpr int kMaxQ = 4;             // query-image buffers
constexpr int kMaxLand = 4;          // landing tiles per epilogue group
constexpr int kMaxClasses = 16;      // slab classes, at most
constexpr int kTmemCols = 512;
constexpr int kSmemBudget = 227 * 1024;
constexpr unsigned long long kTimeoutNs = 4000000000ull;   // 4 s per wait

// Limit of the waits on other CTAs' exchange entries (the merge warps' reads
// of the statistics partials, the fetch warp's reads of lse): kTimeoutNs
// unless a test lowers it (sp_test_set_exchange_wait_ns).  The waits inside
// a CTA, and the drain of its in-flight copies and MMAs, always keep kTimeoutNs.
std::atomic<unsigned long long> g_exchange_wait_ns{kTimeoutNs};

struct TcParams {
    int L, H, H_kv, G, N, R, d;   // N: look-ahead steps of this pass (R = N * G query rows)
    int S;              // slabs = L * H_kv
    int P;              // CTAs
    int F;              // slab classes: CTA c takes slabs s = c % F, c % F + F, ...
    int Pc;             // CTAs per class (P = F * Pc), one token range each
    int U;              // 32-token units of the prompt
    int n_tiles_max;
    int land;           // landing tiles per epilogue group
    int tiles_per_group;  // tiles of one slab an epilogue group takes, at most
    int held;           // held slabs (lag + 1)
    int lag;            // slabs between a slab's P1 and its P2
    int held_base;      // first TMEM column of the held regions
    int stages;
    int nq;             // query-image buffers (2 or 4)
    int64_t T;          // tokens of the prompt (M)
    int64_t slab_stride;  // rows between consecutive slabs in K (the packed token count)
    int64_t tok0;       // row of the prompt's first token within a slab (its offset in the pack)
    int first;          // 1 for the call's first prompt: its preparation clears the status
    int lse_mode;       // 1: each row's lse is given (lse_in); no statistics pass, no exchange
    int la_shift;       // row j sees look-ahead keys 0..j - la_shift
    const float* lse_in;  // [L, H, N] natural-log softmax normalisers (lse_mode)
    float scale, scale_log2e;
    unsigned long long xwait_ns;    // limit of a wait on other CTAs' exchange entries
    // shared-memory carve (byte offsets from the 1024-aligned base)
    int off_q, off_acc, off_c, off_ref, off_stats, off_lse, off_bar, smem_bytes;
    // workspace
    const uint8_t* qimg;            // [S][kRP * d] bf16, 128B-swizzled image of the slab's query rows
    const float2* la;               // [S][kRP] softmax statistics of the look-ahead keys
    unsigned long long* partials;   // [S][kRP][P] (m, z) as 64-bit words; 0 = not yet published
    unsigned long long* lse;        // [S][kRP] (lse bits, tag 1); 0 = not yet published
    WsHeader* hdr;
    float* importance;
    unsigned* acc_glob;             // [N][T] order-preserving codes of the combined maxima (F > 1)
    int* arrivals;                  // [Pc] CTAs of a range done with their maxima (F > 1)
    const __nv_bfloat16* Qp;        // the prompt's look-ahead queries [N, L, H, d] (preparation)
    const __nv_bfloat16* Klap;      // its look-ahead keys [L, H_kv, N_total - la_shift, d] (preparation)
    int N_total, j0;    // all steps of the call; this pass takes steps j0 .. j0 + N - 1
    int accumulate;     // 1: add this pass's share of the mean to importance (passes after the first)
    int Gr;             // query heads per KV head; G (>= Gr, a power of two) query rows per step, the
                        // rows past Gr of each step are zero padding that P2 leaves out
};

// Prompts of one batched launch ("wave"): prompt b owns CTAs [cta0[b], cta0[b+1])
// and has its own plan and workspace slice.
constexpr int kMaxWave = 32;
struct TcBatch {
    int nb;
    int cta0[kMaxWave + 1];
    TcParams p[kMaxWave];
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may stay suspended (without issuing) for up
// to `hint_ns` while the phase is incomplete; it resumes when the phase
// completes.  Waiting threads then take no issue slots from the working warps.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `parity` to complete.  Returns false if the
// kernel is aborting or the wait timed out (then the abort flag is raised).
// Every waiter consumes a barrier's phases in order, and the producer of phase
// k + 1 first needs every waiter's hand-off of phase k, so a waiter is never
// more than one phase ahead of the barrier.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag, WsHeader* hdr,
                                            int where) {
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_suspend(bar, parity, 1000u)) return true;
        if (*abort_flag) return false;
        if (global_ns() - t0 > kTimeoutNs) {
            record_error(hdr, SP_ETIMEOUT, where);
            *abort_flag = 1;
            return false;
        }
    }
}

// The common case (the phase already completed) stays inline: the single-lane
// TMA and MMA issuers share their SM sub-partitions with busy epilogue warps.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, WsHeader* hdr,
                                          int where) {
    return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, abort_flag, hdr, where);
}

__device__ __forceinline__ unsigned long long ld_cg64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.global.cg.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long pack2(float a, float b) {
    return (unsigned long long)__float_as_uint(a) | ((unsigned long long)__float_as_uint(b) << 32);
}

__device__ __forceinline__ float2 unpack2(unsigned long long v) {
    return make_float2(__uint_as_float((unsigned)(v & 0xffffffffu)), __uint_as_float((unsigned)(v >> 32)));
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Named barriers: 3 = the eight epilogue warps (once, at the end), 4 = merge warps.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 3, 512;" ::: "memory"); }
__device__ __forceinline__ void merge_sync() { asm volatile("bar.sync 4, 128;" ::: "memory"); }

// Barrier over `count` threads that also returns whether any of them passed
// `c`: a stop decision taken from it is the same in every thread, so no thread
// goes on to a barrier that the others have left.
__device__ __forceinline__ bool bar_any(int id, int count, bool c) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 q, %2, 0;\n\t"
        "bar.red.or.pred p, %1, %3, q;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(r)
        : "r"(id), "r"((int)c), "r"(count)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool merge_sync_any(bool c) { return bar_any(4, 128, c); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);     // start address
    d |= (uint64_t)1u << 16;                      // leading-dimension byte offset (unused with this swizzle)
    d |= (uint64_t)(1024u >> 4) << 32;            // stride-dimension byte offset
    d |= (uint64_t)1u << 46;                      // descriptor version
    d |= (uint64_t)2u << 61;                      // 128-byte swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B (K-major),
// fp32 accumulator, M = 128, N = n.
__host__ __device__ constexpr uint32_t instr_desc_bf16(int n) {
    return (1u << 4)                    // accumulator format: f32
           | (1u << 7)                  // A format: bf16
           | (1u << 10)                 // B format: bf16
           | ((uint32_t)(n >> 3) << 17) // N / 8
           | ((uint32_t)(128 >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane, as floats.
__device__ __forceinline__ void tmem_ld16f(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 8 consecutive 32-bit columns of this thread's TMEM lane, in two steps: the
// load is issued, and the registers may be used only after tmem_ld8_wait (it
// takes them as operands, so no use can be scheduled above it).
__device__ __forceinline__ void tmem_ld8_issue(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld8_wait(uint32_t (&r)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
                 :
                 : "memory");
}

// Asynchronous store of 8 columns (the registers are read when it issues);
// tmem_wait_st() before the columns are read again.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}

// 16 consecutive floats from a 16-byte aligned shared-memory address.
__device__ __forceinline__ void load16(const float* src, float (&v)[16]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float4 f = reinterpret_cast<const float4*>(src)[k];
        v[4 * k] = f.x; v[4 * k + 1] = f.y; v[4 * k + 2] = f.z; v[4 * k + 3] = f.w;
    }
}

// Row results of 16 values per lane over the warp's 32 lanes (maximum or sum)
// by a halving butterfly: on return lanes 2r and 2r + 1 hold row r's.  A lane
// with `take` false contributes -inf (maximum) or 0 (sum).
template <bool kMax>
__device__ __forceinline__ float warp_rows16(const float (&v)[16], bool take) {
    const int lane = threadIdx.x & 31;
    auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
    const float none = kMax ? -INFINITY : 0.f;
    float a8[8], a4[4], a2[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float lo = take ? v[k] : none, hi = take ? v[k + 8] : none;
        a8[k] = op(b4 ? hi : lo, __shfl_xor_sync(0xffffffffu, b4 ? lo : hi, 16));
    }
#pragma unroll
    for (int k = 0; k < 4; ++k)
        a4[k] = op(b3 ? a8[k + 4] : a8[k], __shfl_xor_sync(0xffffffffu, b3 ? a8[k] : a8[k + 4], 8));
#pragma unroll
    for (int k = 0; k < 2; ++k)
        a2[k] = op(b2 ? a4[k + 2] : a4[k], __shfl_xor_sync(0xffffffffu, b2 ? a4[k] : a4[k + 2], 4));
    float a1 = op(b1 ? a2[1] : a2[0], __shfl_xor_sync(0xffffffffu, b1 ? a2[0] : a2[1], 2));
    return op(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
}

// A token's running maxima of the look-ahead steps rh*(16/G) .. + 16/G - 1
// (steps past N read as 0, never used).
template <int G>
__device__ __forceinline__ void load_acc(const float* a, int rh, int N, float (&v)[16 / G]) {
#pragma unroll
    for (int jl = 0; jl < 16 / G; ++jl) {
        const int jj = rh * (16 / G) + jl;
        v[jl] = jj < N ? a[jj * kTileRows] : 0.f;
    }
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// y = f32(h) + c for both halves h of a packed fp16 pair: the mixed-precision
// add of sm_100 and later, one instruction per half.  The widening is exact,
// so the result is the fp32 sum rounded once, as with a conversion first.
__device__ __forceinline__ void add_h2_f32(uint32_t h2, float c0, float c1, float& y0, float& y1) {
    asm("{\n\t.reg .f16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "add.rn.f32.f16 %0, lo, %3;\n\tadd.rn.f32.f16 %1, hi, %4;\n\t}"
        : "=f"(y0), "=f"(y1) : "r"(h2), "f"(c0), "f"(c1));
}

// max(a, b, c) in one instruction (three-input max of sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// m = max(m, y[0], ..., y[G-1])
template <int G>
__device__ __forceinline__ float fold_heads(float m, const float* y) {
#pragma unroll
    for (int hh = 0; hh + 1 < G; hh += 2) m = fmax3(m, y[hh], y[hh + 1]);
    if (G & 1) m = fmaxf(m, y[G - 1]);
    return m;
}

// m = max(m, y[0], ..., y[gr-1]) for the first gr of G values (the rest are padding rows)
template <int G>
__device__ __forceinline__ float fold_heads_masked(float m, const float* y, int gr) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh)
        if (hh < gr) m = fmaxf(m, y[hh]);
    return m;
}

// Order-preserving 32-bit code of a float (a < b  <=>  code(a) < code(b) as
// unsigned), so that atomicMax on codes takes the max of floats; 0 is below
// the code of every float.
__device__ __forceinline__ unsigned order_code(float x) {
    const unsigned b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float order_decode(unsigned c) {
    return __uint_as_float((c & 0x80000000u) ? (c ^ 0x80000000u) : ~c);
}

// Merge softmax statistics (m2, z2) into (m, z) (natural-log domain).
__device__ __forceinline__ void merge(float& m, float& z, float m2, float z2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) { m = m2; z = z2; return; }
    const float mx = fmaxf(m, m2);
    z = z * ex2_approx(m - mx) + z2 * ex2_approx(m2 - mx);
    m = mx;
}

// ---------------------------------------------------------------------------
// Per-call preparation (one block per slab): the swizzled query image, the
// softmax statistics of the look-ahead keys, and the zeroed exchange entries
// (a zero word means "not published yet"); block 0 of the call's first prompt
// also clears the status.
// ---------------------------------------------------------------------------

// Block s (one per slab) of one prompt's preparation.
template <int KB, int HV>
__device__ __forceinline__ void tc_prep_body(const TcParams& p, int s) {
    const __nv_bfloat16* __restrict__ Q = p.Qp;
    const __nv_bfloat16* __restrict__ Kla = p.Klap;
    uint8_t* __restrict__ qimg = const_cast<uint8_t*>(p.qimg);
    float2* __restrict__ la = const_cast<float2*>(p.la);
    unsigned long long* __restrict__ lse = p.lse;
    unsigned long long* __restrict__ partials = p.partials;
    WsHeader* hdr = p.hdr;
    const int l = s / p.H_kv, g = s % p.H_kv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Loads first (the query rows of the image, then the look-ahead dot
    // products), stores after, so that the load latencies overlap.
    const int cpr = p.d / 8;                      // 16-byte chunks per row
    uint8_t* img = qimg + (size_t)s * kRP * p.d * 2;
    uint4 iv[2];                                  // at most 32 rows x 16 chunks over 256 threads
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int idx = threadIdx.x + u * (int)blockDim.x, r = idx / cpr, ch = idx % cpr;
        iv[u] = make_uint4(0u, 0u, 0u, 0u);
        if (idx < kRP * cpr && r < p.R && r % p.G < p.Gr) {
            const int j = r / p.G, h = g * p.Gr + r % p.G;
            iv[u] = *reinterpret_cast<const uint4*>(Q + (((size_t)j * p.L + l) * p.H + h) * p.d + ch * 8);
        }
    }
    // row r (query j = r / G, head g*Gr + r % G) against look-ahead keys
    // k <= j0 + j - shift: eight consecutive lanes per row, each with an
    // eighth of every dot product (HV = d / 64 16-byte chunks: sub, sub + 8),
    // the keys KB at a time with all their loads in flight, the eight parts added by
    // shuffles; every lane of the row then holds the row's statistics
    if (!p.lse_mode) {
        const int nk = p.N_total - p.la_shift;        // look-ahead keys stored per (layer, KV head)
        const int sub = lane & 7;
        for (int r0 = warp * 4; r0 < kRP; r0 += (blockDim.x / 32) * 4) {
            const int r = r0 + (lane >> 3);
            const bool real = r < p.R && r % p.G < p.Gr;
            const int j = r / p.G, h = g * p.Gr + r % p.G;          // step j0 + j of the call
            const int nkeys = real ? max(0, p.j0 + j - p.la_shift + 1) : 0;
            int kmax = nkeys;                                         // the warp's longest key list
#pragma unroll
            for (int o = 8; o < 32; o <<= 1) kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
            uint4 qa[HV];
#pragma unroll
            for (int t = 0; t < HV; ++t) qa[t] = make_uint4(0u, 0u, 0u, 0u);
            if (real) {
                const uint4* q = reinterpret_cast<const uint4*>(Q + (((size_t)j * p.L + l) * p.H + h) * p.d);
#pragma unroll
                for (int t = 0; t < HV; ++t) qa[t] = q[sub + 8 * t];
            }
            const uint4* kbase = reinterpret_cast<const uint4*>(Kla + ((size_t)l * p.H_kv + g) * nk * p.d);
            float m = -INFINITY, z = 0.f;
            for (int k0 = 0; k0 < kmax; k0 += KB) {
                uint4 kb[KB][HV];
#pragma unroll
                for (int kk = 0; kk < KB; ++kk)
#pragma unroll
                    for (int t = 0; t < HV; ++t)
                        kb[kk][t] = k0 + kk < nkeys
                                        ? kbase[(size_t)(k0 + kk) * (p.d / 8) + sub + 8 * t]
                                        : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int kk = 0; kk < KB; ++kk) {
                    float u = 0.f;
#pragma unroll
                    for (int t = 0; t < HV; ++t) {
                        const uint32_t aw[4] = {qa[t].x, qa[t].y, qa[t].z, qa[t].w};
                        const uint32_t bw[4] = {kb[kk][t].x, kb[kk][t].y, kb[kk][t].z, kb[kk][t].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {         // a bf16 pair widens exactly by shifts
                            u = fmaf(__uint_as_float(aw[e] << 16), __uint_as_float(bw[e] << 16), u);
                            u = fmaf(__uint_as_float(aw[e] & 0xffff0000u), __uint_as_float(bw[e] & 0xffff0000u), u);
                        }
                    }
#pragma unroll
                    for (int o = 1; o < 8; o <<= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
                    if (k0 + kk < nkeys) merge(m, z, u * p.scale_log2e, 1.f);
                }
            }
            if (sub == 0 && r < kRP) la[(size_t)s * kRP + r] = make_float2(m, z);
        }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int idx = threadIdx.x + u * (int)blockDim.x, r = idx / cpr, ch = idx % cpr;
        if (idx < kRP * cpr) {
            const int half = ch >> 3, c = ch & 7;
            const size_t off = (size_t)half * (kRP * 128) + (size_t)r * 128 + (size_t)((c ^ (r & 7)) * 16);
            *reinterpret_cast<uint4*>(img + off) = iv[u];
        }
    }
    if (p.first && s == 0 && threadIdx.x < (int)(sizeof(WsHeader) / 4)) reinterpret_cast<int32_t*>(hdr)[threadIdx.x] = 0;
    if (p.lse_mode) {
        // the given lse, already published (tag 1) for the fetch warp; padded rows 0
        if (threadIdx.x < kRP) {
            const int r = threadIdx.x;
            float v = 0.f;
            if (r < p.R && r % p.G < p.Gr)
                v = p.lse_in[((size_t)l * p.H + g * p.Gr + r % p.G) * p.N_total + p.j0 + r / p.G] *
                    1.4426950408889634f;
            lse[(size_t)s * kRP + r] = (unsigned long long)__float_as_uint(v) | (1ull << 32);
        }
    } else {
        if (threadIdx.x < kRP) lse[(size_t)s * kRP + threadIdx.x] = 0ull;
        unsigned long long* ps = partials + (size_t)s * kRP * p.Pc;
        for (int i = threadIdx.x; i < kRP * p.Pc; i += blockDim.x) ps[i] = 0ull;
    }
    if (p.F > 1) {
        // combined running maxima (0 is below every encoded float) and the
        // per-range arrival counters
        const size_t n = (size_t)p.N * p.T;
        for (size_t i = (size_t)s * blockDim.x + threadIdx.x; i < n; i += (size_t)p.S * blockDim.x)
            p.acc_glob[i] = 0u;
        for (int i = s * blockDim.x + threadIdx.x; i < p.Pc; i += p.S * blockDim.x) p.arrivals[i] = 0;
    }
}

// One call (HV = d / 64): two blocks per SM, up to 128 registers a thread for
// eight keys in flight; a call's 256 or so slabs run in one round.
template <int HV>
__global__ void __launch_bounds__(256, 2) tc_prep_kernel(const __grid_constant__ TcParams p) {
    tc_prep_body<8, HV>(p, blockIdx.x);
}

// All prompts of a wave: blocks b * S .. b * S + S - 1 prepare prompt b; four
// blocks per SM (64 registers a thread: four keys in flight at d = 64, two at
// d = 128), so that a wave's several hundred slabs run in one or two rounds.
template <int HV>
__global__ void __launch_bounds__(256, 4) tc_prep_batch_kernel(const __grid_constant__ TcBatch bt) {
    const int S = bt.p[0].S;
    tc_prep_body<4 / HV, HV>(bt.p[blockIdx.x / S], blockIdx.x % S);
}

// ---------------------------------------------------------------------------
// The persistent scoring kernel
// ---------------------------------------------------------------------------

// Every lane of the warp tests the barrier phase (no divergent branch on the
// common path); a vote makes the outcome the warp's, which then leaves or goes
// on together.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, WsHeader* hdr,
                                          int where) {
    const bool ok = mbar_wait(bar, parity, abort_flag, hdr, where);
    return __all_sync(0xffffffffu, ok);
}

// K viewed as a 2D tensor of rows by d bf16 columns, in 64-column boxes of 128
// rows (a full tile per copy) and of 32 rows (a slab's ragged last tile).
struct KMaps {
    CUtensorMap full, tail;
};

template <int D, int G>
__device__ __forceinline__ void tc_score_body(const KMaps& kmaps, const TcParams& p, const int c) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by pointer arithmetic on the shared array (a round trip
    // through an integer would leave the compiler generic addressing for every
    // shared-memory access: 7% more instructions per tile)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr int kHalves = D / 64;
    constexpr int kStageBytes = kTileRows * D * 2;
    constexpr int kQBytes = kRP * D * 2;
    constexpr uint32_t kIdesc = instr_desc_bf16(kRP);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Slab class and token range of this CTA: it takes slabs s = cf, cf + F, ...
    // (n_slabs of them) over the tokens [t_begin, t_end) of each.  The F CTAs
    // with the same range combine their running maxima at the end.
    const int cf = c % p.F, cr = c / p.F;
    const int n_slabs = (p.S - cf + p.F - 1) / p.F;
    const int u0 = (int)(((int64_t)cr * p.U) / p.Pc), u1 = (int)(((int64_t)(cr + 1) * p.U) / p.Pc);
    const int64_t t_begin = (int64_t)u0 * kUnit;
    const int64_t t_end = min((int64_t)u1 * kUnit, p.T);
    const int len = (int)(t_end - t_begin);
    const int n_tiles = (len + kTileRows - 1) / kTileRows;

    uint8_t* k_stage = smem;                                       // [stages][kStageBytes]
    uint8_t* q_buf = smem + p.off_q;                               // [nq][kQBytes]
    float* acc = reinterpret_cast<float*>(smem + p.off_acc);       // [2 groups][n_tiles_max][N][128]
    float* cbuf = reinterpret_cast<float*>(smem + p.off_c);        // [2 groups][held][tiles_per_group][4][kRP]
    float* rbuf = reinterpret_cast<float*>(smem + p.off_ref);      // [16 epilogue warps][16]
    float2* stats = reinterpret_cast<float2*>(smem + p.off_stats); // [kStatsRing][2 groups][4][kRP]
    float* lse_ring = reinterpret_cast<float*>(smem + p.off_lse);  // [kRing][kRP]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint64_t* k_full = bars;
    uint64_t* k_empty = bars + p.stages;
    uint64_t* q_full = bars + 2 * p.stages;        // [kMaxQ]
    uint64_t* q_empty = q_full + kMaxQ;
    uint64_t* land_full = q_empty + kMaxQ;         // [2 groups][kMaxLand]
    uint64_t* land_empty = land_full + 2 * kMaxLand;
    uint64_t* stats_full = land_empty + 2 * kMaxLand;   // [kStatsRing]
    uint64_t* stats_empty = stats_full + kStatsRing;
    uint64_t* lse_full = stats_empty + kStatsRing; // [kRing]
    uint64_t* lse_empty = lse_full + kRing;
    uint64_t* final_bar = lse_empty + kRing;
    volatile uint32_t* tmem_base_sh = reinterpret_cast<volatile uint32_t*>(final_bar + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_base_sh + 1);
    volatile int* published = abort_flag + 1;      // slabs this CTA has published
    volatile int* last_flag = published + 1;       // this CTA completes its token range (F > 1)

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(smem_u32(&k_full[i]), 1);
            mbar_init(smem_u32(&k_empty[i]), 1);
        }
        for (int i = 0; i < kMaxQ; ++i) {
            mbar_init(smem_u32(&q_full[i]), 1);
            mbar_init(smem_u32(&q_empty[i]), 1);
        }
        for (int i = 0; i < 2 * kMaxLand; ++i) {
            mbar_init(smem_u32(&land_full[i]), 1);
            mbar_init(smem_u32(&land_empty[i]), kEpiWarpsPerGroup);   // one arrival per epilogue warp of the group
        }
        for (int i = 0; i < kStatsRing; ++i) {
            mbar_init(smem_u32(&stats_full[i]), 2 * kEpiWarpsPerGroup);   // every epilogue warp
            mbar_init(smem_u32(&stats_empty[i]), 1);
        }
        for (int i = 0; i < kRing; ++i) {
            mbar_init(smem_u32(&lse_full[i]), 1);
            mbar_init(smem_u32(&lse_empty[i]), 2 * kEpiWarpsPerGroup);
        }
        mbar_init(smem_u32(final_bar), 1);
        *abort_flag = 0;
        *published = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32((const void*)tmem_base_sh)), "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // running max of (s - lse) over (layer, head), per token and look-ahead step
    for (int i = threadIdx.x; i < 2 * p.n_tiles_max * p.N * kTileRows; i += kThreads) acc[i] = -INFINITY;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_base_sh;

    // Every CTA streams its tiles in plain order: slab after slab, the slab's
    // tiles in order (k = s * n_tiles + t).  Tile k goes to epilogue group k % 2,
    // so both groups work on every slab and the HBM stream stays sequential.
    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            int it = 0;
            int st = 0, st_round = 0;          // it % stages, it / stages
            bool ok = true;
            for (int i = 0; i < n_slabs && ok; ++i) {
                const int s = cf + i * p.F, qb = i % p.nq;
                if (i >= p.nq) ok = mbar_wait(smem_u32(&q_empty[qb]), ((i / p.nq) - 1) & 1, abort_flag, p.hdr, 1);
                if (!ok) break;
                mbar_expect_tx(smem_u32(&q_full[qb]), kQBytes);
                bulk_load(smem_u32(q_buf + qb * kQBytes), p.qimg + (size_t)s * kQBytes, kQBytes,
                          smem_u32(&q_full[qb]));
                const int64_t row0 = (int64_t)s * p.slab_stride + p.tok0 + t_begin;
                for (int t = 0; t < n_tiles; ++t, ++it) {
                    if (st_round > 0)
                        ok = mbar_wait(smem_u32(&k_empty[st]), (st_round - 1) & 1, abort_flag, p.hdr, 2);
                    if (!ok) break;
                    const int rows = min(kTileRows, len - t * kTileRows);
                    const uint32_t dst = smem_u32(k_stage + (size_t)st * kStageBytes);
                    const uint32_t bar = smem_u32(&k_full[st]);
                    const int y = (int)(row0 + t * kTileRows);
                    if (rows == kTileRows) {
                        mbar_expect_tx(bar, (uint32_t)(kTileRows * D * 2));
#pragma unroll
                        for (int hf = 0; hf < kHalves; ++hf)
                            tma_load_2d(dst + hf * (kTileRows * 128), &kmaps.full, hf * 64, y, bar);
                    } else {
                        const int nbox = (rows + kBoxRows - 1) / kBoxRows;
                        mbar_expect_tx(bar, (uint32_t)(nbox * kBoxRows * D * 2));
                        for (int hf = 0; hf < kHalves; ++hf)
                            for (int b = 0; b < nbox; ++b)
                                tma_load_2d(dst + hf * (kTileRows * 128) + b * (kBoxRows * 128), &kmaps.tail, hf * 64,
                                            y + b * kBoxRows, bar);
                    }
                    if (++st == p.stages) {
                        st = 0;
                        ++st_round;
                    }
                }
            }
            // wait (bounded) for every copy still in flight before the CTA may exit
            for (int j = max(0, it - p.stages); j < it; ++j) {
                const unsigned long long t0 = global_ns();
                while (!mbar_try_wait(smem_u32(&k_full[j % p.stages]), (j / p.stages) & 1))
                    if (global_ns() - t0 > kTimeoutNs) break;
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            int st = 0, st_round = 0;          // the tile's stage and how often the ring wrapped
            int g = 0;                         // epilogue group of the tile (tiles alternate)
            int ls0 = 0, lr0 = 0, ls1 = 0, lr1 = 0;   // per group: landing slot, wraps of its ring
            bool ok = true;
            for (int i = 0; i < n_slabs && ok; ++i) {
                const int qb = i % p.nq;
                ok = mbar_wait(smem_u32(&q_full[qb]), (i / p.nq) & 1, abort_flag, p.hdr, 4);
                if (!ok) break;
                // descriptors of the K-major operands advance by constant offsets
                const uint64_t b0 = smem_desc(smem_u32(q_buf + qb * kQBytes));
                for (int t = 0; t < n_tiles; ++t) {
                    const int ls = g ? ls1 : ls0, lr = g ? lr1 : lr0;
                    const int slot = g * p.land + ls;
                    ok = mbar_wait(smem_u32(&k_full[st]), st_round & 1, abort_flag, p.hdr, 5);
                    if (ok && lr > 0) ok = mbar_wait(smem_u32(&land_empty[slot]), (lr - 1) & 1, abort_flag, p.hdr, 3);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t a0 = smem_desc(smem_u32(k_stage + (size_t)st * kStageBytes));
                    const uint32_t d_tmem = tmem_base + (uint32_t)(slot * kRP);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const int hf = kk >> 2, ko = kk & 3;
                        tc_mma(d_tmem, a0 + (uint64_t)((hf * (kTileRows * 128) + ko * 32) >> 4),
                               b0 + (uint64_t)((hf * (kRP * 128) + ko * 32) >> 4), kIdesc, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&k_empty[st]));
                    tc_commit(smem_u32(&land_full[slot]));
                    if (++st == p.stages) {
                        st = 0;
                        ++st_round;
                    }
                    const int ls_n = ls + 1 == p.land ? 0 : ls + 1, lr_n = ls + 1 == p.land ? lr + 1 : lr;
                    if (g) { ls1 = ls_n; lr1 = lr_n; } else { ls0 = ls_n; lr0 = lr_n; }
                    g ^= 1;
                }
                if (!ok) break;
                tc_commit(smem_u32(&q_empty[qb]));
            }
            // all MMAs issued so far complete before TMEM may be freed
            tc_commit(smem_u32(final_bar));
            const unsigned long long t0 = global_ns();
            while (!mbar_try_wait(smem_u32(final_bar), 0))
                if (global_ns() - t0 > kTimeoutNs) break;
        }
        __syncwarp();
    } else if (warp < kPubWarp) {
        // ------------------------------ epilogue ------------------------------
        // Sixteen warps, two groups of eight; group g takes the tiles k with
        // k % 2 == g (k = s * n_tiles + t), so both groups work on every slab.
        // A warp owns one TMEM lane quadrant (32 tokens of every tile) and one
        // half of the query rows (16 of the 32 columns), and works on it alone:
        // statistics and fp16 references are per (quadrant, row), and the
        // hand-offs to the other roles are mbarriers that count the warps taking
        // part, so no warp ever waits at a barrier for another.
        const int ew = warp - 2;                       // 0..15
        const int grp = ew >> 3;
        const int quad = warp & 3;                     // TMEM lane quadrant of this warp
        const int rh = (ew >> 2) & 1;                  // query rows rh*16 .. rh*16 + 15
        const int tok = quad * 32 + lane;              // token row inside a tile
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        const int tpg = p.tiles_per_group;             // held tile slots per slab
        float* acc_g = acc + (size_t)grp * p.n_tiles_max * p.N * kTileRows;
        float* cb_g = cbuf + (size_t)grp * p.held * tpg * 4 * kRP;
        float* wref = rbuf + ew * 16;                  // the warp's 16 row references (P1)
        const uint32_t held_g = tmem_base + lane_addr + (uint32_t)(p.held_base + grp * p.held * tpg * 16 + rh * 8);
        const int odd = n_tiles & 1;
        const bool all_rows = p.R == kRP && p.Gr == G;  // every query row is a real (step, head) row
        int ls = 0, lph = 0;                           // next landing tile of the group's ring, its phase
        int hs1 = 0, hs2 = 0;                          // held slots of the next P1 and P2 slabs
        uint32_t chg = 0;                              // held tiles (hs * tpg + j) whose references P2 reloads
        bool ok = true;
        if (p.lse_mode) {
            // lse given: one pass, exp(s - lse) straight from the landing tiles
            for (int i = 0; i < n_slabs && ok; ++i) {
                const int q = i % kRing, t0 = (grp + i * odd) & 1;
                if (!warp_wait(smem_u32(&lse_full[q]), (i / kRing) & 1, abort_flag, p.hdr, 8)) {
                    ok = false;
                    break;
                }
                float lr[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) lr[r] = lse_ring[q * kRP + rh * 16 + r];
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&lse_empty[q]));
                for (int t = t0; t < n_tiles; t += 2) {
                    const int slot = grp * p.land + ls;
                    if (!warp_wait(smem_u32(&land_full[slot]), lph, abort_flag, p.hdr, 6)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    float x[16];
                    tmem_ld16f(tmem_base + lane_addr + (uint32_t)(slot * kRP + rh * 16), x);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&land_empty[slot]));
                    if (++ls == p.land) { ls = 0; lph ^= 1; }
                    float* a = acc_g + (size_t)t * p.N * kTileRows + tok;
#pragma unroll
                    for (int jl = 0; jl < 16 / G; ++jl) {
                        const int jj = rh * (16 / G) + jl;
                        if (jj < p.N) {
                            float y[G];
#pragma unroll
                            for (int hh = 0; hh < G; ++hh) y[hh] = fmaf(x[jl * G + hh], p.scale_log2e, -lr[jl * G + hh]);
                            a[jj * kTileRows] = p.Gr == G ? fold_heads<G>(a[jj * kTileRows], y)
                                                          : fold_heads_masked<G>(a[jj * kTileRows], y, p.Gr);
                        }
                    }
                }
            }
        }
        for (int i = 0; i < (p.lse_mode ? 0 : n_slabs + p.lag) && ok; ++i) {
            // ---- P1: statistics of this CTA's i-th slab over the group's tiles, as fp16 offsets ----
            if (i < n_slabs) {
                const int s = i, q = s % kStatsRing, hs = hs1;
                if (++hs1 == p.held) hs1 = 0;
                const int t0 = (grp + s * odd) & 1;    // this group's first tile of the slab
                if (s >= kStatsRing &&
                    !warp_wait(smem_u32(&stats_empty[q]), ((s / kStatsRing) - 1) & 1, abort_flag, p.hdr, 7)) {
                    ok = false;
                    break;
                }
                // Statistics of query row rh*16 + r over this quadrant's tokens,
                // relative to a reference ref[r] that the whole warp shares: each
                // lane adds its token's exp(s - ref) of every row to its own
                // running sums zacc[r], and the 32 lanes' sums of a row are added
                // once, at the end of the slab (lanes 2r, 2r + 1).  The reference
                // starts at the row's maximum over the slab's first tile with a
                // valid token and rises to a tile's maximum whenever a logit
                // exceeds it by more than kRefMargin (every lane's sums of that
                // row are then rescaled).  It is always a logit of the row, so
                // z >= 1 once a token was valid, and the held fp16 offsets s - ref
                // stay at most kRefMargin above 0.  Row maxima go through a
                // shuffle butterfly, and a tile's references are stored for P2
                // only when they change: shared memory is slow while the MMA
                // reads its operands.
                float ref_lane = 0.f;                  // ref of row rh*16 + (lane >> 1); all 16 in wref
                float zacc[16];                        // this lane's sums of exp(s - ref), per row
#pragma unroll
                for (int r = 0; r < 16; ++r) zacc[r] = 0.f;
                chg &= ~(((1u << tpg) - 1u) << (hs * tpg));
                // One tile of P1, specialised at compile time for the slab's first
                // tile of this group (it sets the references: no comparison, no
                // rescale) and for full tiles (every lane's token is valid), so
                // the common case -- a later, full tile -- carries no per-value
                // selects or flags.
                auto p1_tile = [&](auto first_c, auto full_c, int t, int j) -> bool {
                    constexpr bool kFirst = decltype(first_c)::value, kFull = decltype(full_c)::value;
                    const int slot = grp * p.land + ls;
                    float ref[16];                     // read while the landing tile is awaited
                    if constexpr (!kFirst) load16(wref, ref);
                    if (!warp_wait(smem_u32(&land_full[slot]), lph, abort_flag, p.hdr, 6)) return false;
                    tc_fence_after();
                    float x[16];
                    tmem_ld16f(tmem_base + lane_addr + (uint32_t)(slot * kRP + rh * 16), x);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&land_empty[slot]));    // this part is read
                    if (++ls == p.land) { ls = 0; lph ^= 1; }
                    const bool valid = kFull || t * kTileRows + tok < len;
                    float o[16];
                    uint32_t pk[8];
                    auto pack_store = [&]() {
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const __half2 h2 = __floats2half2_rn(o[2 * k], o[2 * k + 1]);
                            pk[k] = *reinterpret_cast<const uint32_t*>(&h2);
                        }
                        tmem_st8(held_g + (uint32_t)((hs * tpg + j) * 16), pk);
                    };
                    bool redo = true;
                    if constexpr (kFirst) {
#pragma unroll
                        for (int r = 0; r < 16; ++r) o[r] = x[r] * p.scale_log2e;
                    } else {
#pragma unroll
                        for (int r = 0; r < 16; ++r) o[r] = fmaf(x[r], p.scale_log2e, -ref[r]);
                        const float m0 = fmax3(o[0], o[1], o[2]), m1 = fmax3(o[3], o[4], o[5]);
                        const float m2 = fmax3(o[6], o[7], o[8]), m3 = fmax3(o[9], o[10], o[11]);
                        const float m4 = fmax3(o[12], o[13], o[14]);
                        const float om = fmaxf(fmax3(m0, m1, m2), fmax3(m3, m4, o[15]));
                        redo = __any_sync(0xffffffffu, (kFull || valid) && om > kRefMargin);
                        // the fp16 offsets with the current references go to TMEM
                        // while the vote resolves (stored again if a reference rises)
                        pack_store();
                    }
                    if (redo) {
                        // each reference starts at its row's largest value (first
                        // tile) or rises by the row's largest offset
                        const float mx = warp_rows16<true>(o, valid);   // finite: a lane is valid
                        if constexpr (kFirst) {
                            ref_lane = mx;
#pragma unroll
                            for (int r = 0; r < 16; ++r) o[r] -= __shfl_sync(0xffffffffu, mx, 2 * r);
                        } else {
                            const float dm = fmaxf(mx, 0.f);
                            ref_lane += dm;
                            const float f = ex2_approx(-dm);   // rescale of the row's sums
#pragma unroll
                            for (int r = 0; r < 16; ++r) {
                                o[r] -= __shfl_sync(0xffffffffu, dm, 2 * r);
                                zacc[r] *= __shfl_sync(0xffffffffu, f, 2 * r);
                            }
                        }
                        if ((lane & 1) == 0) wref[lane >> 1] = ref_lane;
                        __syncwarp();
                        // the tile's fp16 references differ from the previous tile's: P2 reloads them
                        const float rr = __shfl_sync(0xffffffffu, ref_lane, 2 * (lane & 15));
                        float* cq = cb_g + (((size_t)hs * tpg + j) * 4 + quad) * kRP + rh * 16;
                        if (lane < 16) cq[lane] = rr;
                        chg |= 1u << (hs * tpg + j);
                        if constexpr (!kFirst) tmem_wait_st();   // the first store has landed before this one
                        pack_store();
                    }
                    if constexpr (kFull) {
#pragma unroll
                        for (int r = 0; r < 16; ++r) zacc[r] += ex2_approx(o[r]);
                    } else {
                        // (the lanes past the range occur only in a ragged last tile)
#pragma unroll
                        for (int r = 0; r < 16; ++r) zacc[r] += valid ? ex2_approx(o[r]) : 0.f;
                    }
                    tmem_wait_st();
                    return true;
                };
                using T_ = std::true_type;
                using F_ = std::false_type;
                const bool have_ref = t0 < n_tiles;    // the group has a tile of this slab
                for (int t = t0, j = 0; t < n_tiles; t += 2, ++j) {
                    const bool full_tile = (t + 1) * kTileRows <= len;
                    bool done;
                    if (j == 0) done = full_tile ? p1_tile(T_{}, T_{}, t, j) : p1_tile(T_{}, F_{}, t, j);
                    else done = full_tile ? p1_tile(F_{}, T_{}, t, j) : p1_tile(F_{}, F_{}, t, j);
                    if (!done) {
                        ok = false;
                        break;
                    }
                }
                if (!ok) break;
                const float z_lane = warp_rows16<false>(zacc, true);   // row (lane >> 1)'s sum over the lanes
                if ((lane & 1) == 0)
                    stats[((q * 2 + grp) * 4 + quad) * kRP + rh * 16 + (lane >> 1)] =
                        make_float2(have_ref ? ref_lane : -INFINITY, z_lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&stats_full[q]));
            }
            // ---- P2: normalise the group's tiles of the (i - lag)-th slab, fold the max ----
            if (i >= p.lag) {
                const int s = i - p.lag, q = s % kRing, hs = hs2;
                if (++hs2 == p.held) hs2 = 0;
                const int t0 = (grp + s * odd) & 1;
                if (!warp_wait(smem_u32(&lse_full[q]), (s / kRing) & 1, abort_flag, p.hdr, 8)) {
                    ok = false;
                    break;
                }
                const float* lq = lse_ring + q * kRP + rh * 16;   // the slot is held until P2 is done
                float d[16];                           // the tile's reference - lse, per row
#pragma unroll
                for (int r = 0; r < 16; ++r) d[r] = 0.f;
                for (int t = t0, j = 0; t < n_tiles; t += 2, ++j) {
                    uint32_t pk[8];
                    tmem_ld8_issue(held_g + (uint32_t)((hs * tpg + j) * 16), pk);
                    // shared-memory reads overlap the TMEM load
                    float* a = acc_g + (size_t)t * p.N * kTileRows + tok;
                    float av[16 / G];
                    if (all_rows) {
#pragma unroll
                        for (int jl = 0; jl < 16 / G; ++jl) av[jl] = a[(rh * (16 / G) + jl) * kTileRows];
                    } else {
                        load_acc<G>(a, rh, p.N, av);
                    }
                    if ((chg >> (hs * tpg + j)) & 1u) {
                        float c[16], l[16];
                        load16(cb_g + (((size_t)hs * tpg + j) * 4 + quad) * kRP + rh * 16, c);
                        load16(lq, l);
#pragma unroll
                        for (int r = 0; r < 16; ++r) d[r] = c[r] - l[r];
                    }
                    tmem_ld8_wait(pk);
                    float y[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) add_h2_f32(pk[k], d[2 * k], d[2 * k + 1], y[2 * k], y[2 * k + 1]);
                    // rows rh*16 + k are look-ahead steps jj = rh*(16/G) + k/G, heads k%G
                    if (all_rows) {
#pragma unroll
                        for (int jl = 0; jl < 16 / G; ++jl)
                            a[(rh * (16 / G) + jl) * kTileRows] = fold_heads<G>(av[jl], y + jl * G);
                    } else {
#pragma unroll
                        for (int jl = 0; jl < 16 / G; ++jl) {
                            const int jj = rh * (16 / G) + jl;
                            if (jj < p.N) a[jj * kTileRows] = fold_heads_masked<G>(av[jl], y + jl * G, p.Gr);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&lse_empty[q]));
            }
        }
        epi_sync();                                    // both groups' running maxima are complete
        // importance of a token: (1/N) sum_j exp(max_{l,h}(s - lse))
        const float inv_n = 1.0f / (float)p.N_total;
        const size_t half = (size_t)p.n_tiles_max * p.N * kTileRows;
        if (p.F == 1) {
            if (!*abort_flag && rh == 0) {
                for (int t = grp; t < n_tiles; t += 2) {
                    const int k = t * kTileRows + tok;
                    if (k < len) {
                        const float* a = acc + (size_t)t * p.N * kTileRows + tok;
                        float sum = 0.f;
                        for (int jj = 0; jj < p.N; ++jj) sum += exp2f(fmaxf(a[jj * kTileRows], a[half + jj * kTileRows]));
                        p.importance[t_begin + k] = (p.accumulate ? p.importance[t_begin + k] : 0.f) + sum * inv_n;
                    }
                }
            }
        } else {
            // fold this CTA's maxima (over its slab class) into the range's
            // combined maxima; the last of the range's F CTAs to arrive turns
            // them into importance
            if (!*abort_flag) {
                for (int t = grp; t < n_tiles; t += 2) {
                    const int k = t * kTileRows + tok;
                    if (k < len) {
                        const float* a = acc + (size_t)t * p.N * kTileRows + tok;
                        for (int jj = rh; jj < p.N; jj += 2)
                            atomicMax(&p.acc_glob[(size_t)jj * p.T + t_begin + k],
                                      order_code(fmaxf(a[jj * kTileRows], a[half + jj * kTileRows])));
                    }
                }
            }
            __threadfence();
            epi_sync();
            if (ew == 0 && lane == 0) *last_flag = atomicAdd(&p.arrivals[cr], 1) == p.F - 1 ? 1 : 0;
            epi_sync();
            if (*last_flag && !*abort_flag && rh == 0) {
                __threadfence();
                for (int t = grp; t < n_tiles; t += 2) {
                    const int k = t * kTileRows + tok;
                    if (k < len) {
                        float sum = 0.f;
                        for (int jj = 0; jj < p.N; ++jj)
                            sum += exp2f(order_decode(__ldcg(&p.acc_glob[(size_t)jj * p.T + t_begin + k])));
                        p.importance[t_begin + k] = (p.accumulate ? p.importance[t_begin + k] : 0.f) + sum * inv_n;
                    }
                }
            }
        }
    } else if (warp == kPubWarp) {
        // ------------------------------ publish ------------------------------
        // lane r merges row r's statistics over the two groups and four
        // quadrants and writes them to global memory as one 64-bit word.
        for (int i = 0; i < (p.lse_mode ? 0 : n_slabs); ++i) {
            const int s = cf + i * p.F, q = i % kStatsRing;
            if (!warp_wait(smem_u32(&stats_full[q]), (i / kStatsRing) & 1, abort_flag, p.hdr, 9)) break;
            float m = -INFINITY, z = 0.f;
#pragma unroll
            for (int part = 0; part < 8; ++part) {
                const float2 v = stats[(q * 8 + part) * kRP + lane];
                merge(m, z, v.x, v.y);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&stats_empty[q]));
            st64(&p.partials[((size_t)s * kRP + lane) * p.Pc + cr], pack2(m, z));
            __syncwarp();
            if (lane == 0) *published = i + 1;      // wakes this CTA's merge warps for slab s if it is theirs
        }
    } else if (warp < kFetchWarp) {
        // ------------------------------ merge ------------------------------
        // The class's i-th slab is merged by its CTA with range i mod Pc, once
        // that CTA has published its own statistics of it (the other CTAs are then
        // a few microseconds from done): the entries are read until all are there.
        const int mi = threadIdx.x - kMergeBase;       // 0..127
        const int r = mi >> 2, part = mi & 3;
        for (int i = cr; i < (p.lse_mode ? 0 : n_slabs); i += p.Pc) {
            const int s = cf + i * p.F;
            if (mi == 0) {
                const unsigned long long t0 = global_ns();
                while (*published <= i) {
                    if (*abort_flag) break;
                    if (global_ns() - t0 > kTimeoutNs) {
                        record_error(p.hdr, SP_ETIMEOUT, 12);
                        *abort_flag = 1;
                        break;
                    }
                    __nanosleep(64);
                }
            }
            if (merge_sync_any(*abort_flag != 0)) break;
            const unsigned long long* src = p.partials + ((size_t)s * kRP + r) * p.Pc;
            const float2 la = __ldcg(&p.la[(size_t)s * kRP + r]);
            float m = -INFINITY, z = 0.f;
            bool ok = true;
            for (int base = part; base < p.Pc && ok; base += 64) {
                // all loads of the batch first (up to 16 in flight per thread)
                unsigned long long v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int cc = base + 4 * k;
                    v[k] = cc < p.Pc ? ld_cg64(src + cc) : 0ull;
                }
                // an entry whose store is not visible yet reads as 0: read the missing
                // ones again, all in flight together
                const unsigned long long t0 = global_ns();
                for (;;) {
                    bool missing = false;
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        if (base + 4 * k < p.Pc && (v[k] >> 32) == 0ull) missing = true;
                    if (!missing) break;
                    if (*abort_flag || global_ns() - t0 > p.xwait_ns) { ok = false; break; }
                    __nanosleep(64);
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        if (base + 4 * k < p.Pc && (v[k] >> 32) == 0ull) v[k] = ld_cg64(src + base + 4 * k);
                }
                float mb = -INFINITY;
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (base + 4 * k < p.Pc) mb = fmaxf(mb, unpack2(v[k]).x);
                float zb = 0.f;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    if (base + 4 * k >= p.Pc) continue;
                    const float2 f = unpack2(v[k]);
                    zb += f.y * ex2_approx(f.x - mb);
                }
                merge(m, z, mb, zb);
            }
            if (!ok) {
                record_error(p.hdr, SP_ETIMEOUT, 13);
                *abort_flag = 1;
            }
#pragma unroll
            for (int o = 1; o <= 2; o <<= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
                const float z2 = __shfl_xor_sync(0xffffffffu, z, o);
                merge(m, z, m2, z2);
            }
            if (part == 0) {
                merge(m, z, la.x, la.y);
                const float lse = m + __log2f(z);     // base 2, like every statistic here
                st64(&p.lse[(size_t)s * kRP + r], (unsigned long long)__float_as_uint(lse) | (1ull << 32));
            }
            merge_sync();
        }
    } else {
        // ------------------------------ fetch ------------------------------
        for (int i = 0; i < n_slabs; ++i) {
            const int s = cf + i * p.F, q = i % kRing;
            bool ok = true;
            if (lane == 0 && i >= kRing) ok = mbar_wait(smem_u32(&lse_empty[q]), ((i / kRing) - 1) & 1, abort_flag, p.hdr, 10);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            __syncwarp();
            if (!ok) break;
            const unsigned long long* src = p.lse + (size_t)s * kRP + lane;
            unsigned long long v = ld_cg64(src);
            const unsigned long long t0 = global_ns();
            while (!__all_sync(0xffffffffu, (v >> 32) == 1ull)) {
                // lane 0 decides, so that the warp leaves the loop together
                int stop = 0;
                if (lane == 0) {
                    if (*abort_flag) stop = 1;
                    else if (global_ns() - t0 > p.xwait_ns) {
                        record_error(p.hdr, SP_ETIMEOUT, 11);
                        *abort_flag = 1;
                        stop = 1;
                    }
                }
                if (__shfl_sync(0xffffffffu, stop, 0)) { ok = false; break; }
                __nanosleep(32);
                v = ld_cg64(src);
            }
            if (!ok) break;
            lse_ring[q * kRP + lane] = __uint_as_float((unsigned)(v & 0xffffffffu));
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&lse_full[q]));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// One prompt: CTA c of p.P.
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1) tc_score_kernel(const __grid_constant__ KMaps kmaps,
                                                                const __grid_constant__ TcParams p) {
    tc_score_body<D, G>(kmaps, p, blockIdx.x);
}

// A wave of prompts: CTA blockIdx.x works for the prompt whose range holds it.
template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1) tc_score_batch_kernel(const __grid_constant__ KMaps kmaps,
                                                                      const __grid_constant__ TcBatch bt) {
    int b = 0;
    while (b + 1 < bt.nb && (int)blockIdx.x >= bt.cta0[b + 1]) ++b;
    tc_score_body<D, G>(kmaps, bt.p[b], (int)blockIdx.x - bt.cta0[b]);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

struct Plan {
    TcParams p;
    size_t off_qimg, off_la, off_partials, off_lse, off_acc_glob, off_arrivals, total;
};

int sm_count_or(int fallback) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return fallback; }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return fallback;
    }
    return n;
}

// Look-ahead steps j0 .. j0 + n - 1 of a call: the query rows of one kernel
// pass.  A call with more than kRP / G steps runs in several passes (each
// streams K once); later passes add their share of the mean to importance.
struct Pass {
    int j0, n;
};

// Query rows per look-ahead step: the heads of a KV group, padded to a power
// of two (1, 2, 4, 8 or 16) so that a 16-row half of the MMA columns holds
// whole steps.
int padded_group(int G) {
    int Gp = 1;
    while (Gp < G) Gp <<= 1;
    return Gp;
}

int steps_per_pass(const ScoreProblem& q) { return kRP / padded_group(q.H / q.H_kv); }

bool shape_ok(const ScoreProblem& q) {
    if (q.dtype != SP_BF16 || q.B < 1 || q.N < 1 || q.max_M < 1) return false;
    if (q.d != 64 && q.d != 128) return false;
    if (q.H / q.H_kv > 16) return false;
    if (q.T < 1 || q.T > (int64_t)INT32_MAX / 4) return false;
    if ((int64_t)q.L * q.H_kv * q.T > (int64_t)INT32_MAX) return false;   // TMA row coordinate
    return true;
}

// Plan for one prompt of M tokens of the problem's shape on up to P_hint CTAs;
// returns false if it does not fit this path.
bool make_plan(const ScoreProblem& q, int64_t M, int P_hint, Pass ps, Plan& out) {
    if (!shape_ok(q) || M < 1 || M > q.max_M) return false;
    const int Gp = padded_group(q.H / q.H_kv);
    if (ps.n < 1 || ps.j0 < 0 || ps.j0 + ps.n > q.N || ps.n * Gp > kRP) return false;
    TcParams& p = out.p;
    p.L = q.L; p.H = q.H; p.H_kv = q.H_kv; p.G = Gp; p.N = ps.n; p.R = ps.n * Gp; p.d = q.d;
    p.Gr = q.H / q.H_kv;
    p.N_total = q.N;
    p.j0 = ps.j0;
    p.accumulate = ps.j0 > 0 ? 1 : 0;
    p.S = q.L * q.H_kv;
    p.T = M;
    p.slab_stride = q.T;
    p.tok0 = 0;
    p.U = (int)((M + kUnit - 1) / kUnit);
    const int P0 = std::max(1, std::min(std::min(P_hint, p.U), kMaxCtas));
    // Slab classes: F classes of P0 / F CTAs; a CTA takes ceil(S / F) slabs
    // of a token range of ceil(U / Pc) units, and the F CTAs of a range merge
    // their maxima at the end.  The plan takes the F with the fewest tiles a
    // CTA runs through, each slab's fixed work (statistics and exchange, the
    // references of its first tiles) counted as half a tile: a part-filled
    // last tile costs as much as a full one, so ranges of whole tiles win
    // (measured at 8K: 11 or 13 classes beat 16 and 10 by 4.5%).  With more
    // than one class a range stays within kMaxTiles tiles (the held slabs
    // that hide the exchange need the TMEM).
    {
        int best_F = 1;
        double best = 0.0;
        for (int F = 1; F <= kMaxClasses && F <= p.S && F <= P0; ++F) {
            const int Pc = P0 / F;
            const int tiles = (((p.U + Pc - 1) / Pc) * kUnit + kTileRows - 1) / kTileRows;
            if (F > 1 && tiles > kMaxTiles) continue;
            const double cost = (double)((p.S + F - 1) / F) * (tiles + 0.5);
            if (F == 1 || cost < best) {
                best = cost;
                best_F = F;
            }
        }
        p.F = best_F;
    }
    p.Pc = P0 / p.F;
    p.P = p.Pc * p.F;
    const int units_max = (p.U + p.Pc - 1) / p.Pc;
    p.n_tiles_max = (units_max * kUnit + kTileRows - 1) / kTileRows;
    if (p.n_tiles_max > kMaxTilesLong) return false;
    // TMEM: per epilogue group `land` fp32 landing tiles (32 columns each) and
    // `held` slabs of its fp16 tiles (16 columns per tile, tiles_per_group tiles
    // per slab); two landing tiles when that still leaves room for two held slabs.
    p.tiles_per_group = (p.n_tiles_max + 1) / 2;
    const int slab_cols = p.tiles_per_group * 16;
    p.lse_mode = q.lse_mode ? 1 : 0;
    p.la_shift = q.la_shift;
    p.lse_in = q.lse_in;
    if (p.lse_mode) {
        // no held logits: all of TMEM holds landing tiles
        p.land = kMaxLand;
        p.held = 0;
        p.lag = 0;
    } else {
        p.land = 2;
        p.held = (kTmemCols / 2 - p.land * kRP) / slab_cols;
        if (p.held < 2) {
            p.land = 1;
            p.held = (kTmemCols / 2 - p.land * kRP) / slab_cols;
        }
        if (p.held < 1) return false;
        p.held = std::min(p.held, kMaxHeld);
        p.lag = p.held - 1;
    }
    p.held_base = 2 * p.land * kRP;               // after both groups' landing tiles
    if (p.held_base + 2 * p.held * slab_cols > kTmemCols) return false;
    if (p.held * p.tiles_per_group > 32) return false;   // one bit per held tile
    p.scale = 1.0f / sqrtf((float)q.d);
    p.scale_log2e = p.scale * 1.4426950408889634f;
    p.xwait_ns = g_exchange_wait_ns.load(std::memory_order_relaxed);
    const int stage_bytes = kTileRows * q.d * 2;
    const int q_bytes = kRP * q.d * 2;
    const int n_bars = 2 * 8 + 2 * kMaxQ + 4 * kMaxLand + 2 * kStatsRing + 2 * kRing + 2;
    const int acc_bytes = 2 * p.n_tiles_max * p.N * kTileRows * 4;   // running max (one per group)
    const int c_bytes = 2 * p.held * p.tiles_per_group * 4 * kRP * 4;   // fp16 references per quadrant
    const int ring_bytes = kStatsRing * 2 * 4 * kRP * 8 + kRing * kRP * 4;
    const int fixed = kRefBytes + acc_bytes + c_bytes + ring_bytes + 16 + n_bars * 8 + 16 + 1024;
    // query images: the TMA loads slab s's image once slab s - nq is done, so
    // with one or two tiles per slab a ring of four keeps it ahead of the K
    // stream; with more tiles two are enough
    p.nq = p.n_tiles_max <= 2 ? kMaxQ : 2;
    p.stages = std::min(6, (kSmemBudget - fixed - p.nq * q_bytes) / stage_bytes);
    if (p.stages < 3 && p.nq > 2) {
        p.nq = 2;
        p.stages = std::min(6, (kSmemBudget - fixed - p.nq * q_bytes) / stage_bytes);
    }
    if (p.stages < 2) return false;
    int off = p.stages * stage_bytes;
    p.off_q = off;
    off += p.nq * q_bytes;
    p.off_acc = off;
    off += acc_bytes;
    p.off_c = off;
    off += c_bytes;
    p.off_ref = off;
    off += kRefBytes;
    p.off_stats = off;
    off += kStatsRing * 2 * 4 * kRP * 8;
    p.off_lse = off;
    off += kRing * kRP * 4;
    off = (off + 15) & ~15;
    p.off_bar = off;
    off += (2 * p.stages + 2 * kMaxQ + 4 * kMaxLand + 2 * kStatsRing + 2 * kRing + 2) * 8 + 16;
    // slack for 1024-byte alignment; more than half of the SM's shared memory, so
    // that one CTA runs per SM (each CTA allocates all 512 TMEM columns)
    p.smem_bytes = std::max(off + 1024, 116 * 1024);
    if (p.smem_bytes > kSmemBudget) return false;
    // workspace (after the 256-byte header)
    Carve cv;
    const size_t S = (size_t)p.S;
    out.off_qimg = cv.take(S * kRP * q.d * 2);
    out.off_la = cv.take(S * kRP * sizeof(float2));
    out.off_lse = cv.take(S * kRP * 8);                    // lse and partials are zeroed per call
    out.off_partials = cv.take(S * kRP * (size_t)kMaxCtas * 8);
    out.off_acc_glob = cv.take((size_t)q.N * (size_t)M * 4);
    out.off_arrivals = cv.take((size_t)kMaxCtas * 4);
    out.total = cv.off;
    return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

// Cooperative launch of `grid` CTAs of `kern` (one prompt or a wave).
template <typename Kern, typename Arg>
sp_status launch_coop(Kern kern, const KMaps& maps, const Arg& arg, int grid, int smem_bytes, cudaStream_t st) {
    SP_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes));
    int per_sm = 0;
    SP_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem_bytes));
    if (per_sm < 1) {
        set_error("sp_score: the tensor-core kernel does not fit on an SM (%d bytes of shared memory)", smem_bytes);
        return SP_EUNSUPPORTED;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps, arg);
    count_launch();
    if (e != cudaSuccess) {
        set_error("sp_score: cooperative launch of %d CTAs failed: %s", grid, cudaGetErrorString(e));
        return SP_ECUDA;
    }
    return SP_OK;
}

template <int D, int G>
sp_status launch_kernel(const KMaps& maps, const TcParams& p, cudaStream_t st) {
    return launch_coop(tc_score_kernel<D, G>, maps, p, p.P, p.smem_bytes, st);
}

template <int D, int G>
sp_status launch_batch(const KMaps& maps, const TcBatch& bt, int smem_bytes, cudaStream_t st) {
    return launch_coop(tc_score_batch_kernel<D, G>, maps, bt, bt.cta0[bt.nb], smem_bytes, st);
}

// The prompt's pointers: its workspace slice starts at w; the status header is
// always the first 256 bytes of the whole workspace.
void bind_prompt(const ScoreProblem& q, int b, bool first, uint8_t* ws, uint8_t* w, Plan& plan) {
    TcParams& p = plan.p;
    p.tok0 = q.cu_M_host[b];
    p.first = first ? 1 : 0;
    p.hdr = reinterpret_cast<WsHeader*>(ws);
    p.qimg = w + plan.off_qimg;
    p.la = reinterpret_cast<const float2*>(w + plan.off_la);
    p.partials = reinterpret_cast<unsigned long long*>(w + plan.off_partials);
    p.lse = reinterpret_cast<unsigned long long*>(w + plan.off_lse);
    p.importance = q.importance + q.cu_M_host[b];
    p.acc_glob = reinterpret_cast<unsigned*>(w + plan.off_acc_glob);
    p.arrivals = reinterpret_cast<int*>(w + plan.off_arrivals);
    p.Qp = static_cast<const __nv_bfloat16*>(q.Q) + ((size_t)b * q.N + p.j0) * q.L * q.H * q.d;
    p.Klap = q.Kla ? static_cast<const __nv_bfloat16*>(q.Kla) + (size_t)b * q.L * q.H_kv * (q.N - q.la_shift) * q.d
                   : nullptr;
    p.lse_in = q.lse_in ? q.lse_in + (size_t)b * q.L * q.H * q.N : nullptr;   // [B, L, H, N]
}

// Waves of a batch: consecutive non-empty prompts, at most kMaxWave of them,
// whose minimum CTA counts (kMaxTiles tiles per CTA and slab) fit on the SMs
// together.  Each prompt gets its minimum plus a share of the spare CTAs in
// proportion to its length, its own plan and its own workspace slice.
struct Wave {
    std::vector<int> prompts;
    std::vector<Plan> plans;
    std::vector<size_t> offs;   // workspace slice of each prompt
    size_t bytes = 0;           // the wave's workspace
    int smem = 0;               // the largest plan's shared memory
};

bool plan_waves(const ScoreProblem& q, int sms, Pass ps, std::vector<Wave>& waves) {
    waves.clear();
    const int64_t per_cta = (int64_t)kMaxTiles * kTileRows;      // tokens of a slab one CTA can take
    auto len = [&](int b) { return q.cu_M_host[b + 1] - q.cu_M_host[b]; };
    auto min_ctas = [&](int b) { return (int)((len(b) + per_cta - 1) / per_cta); };
    std::vector<int> cur;
    int64_t tot = 0;
    int need = 0;
    auto flush = [&]() -> bool {
        if (cur.empty()) return true;
        Wave w;
        w.prompts = cur;
        const int n = (int)cur.size();
        std::vector<int> P(n);
        const int spare = sms - need;
        int used = 0;
        for (int i = 0; i < n; ++i) {
            P[i] = min_ctas(cur[i]) + (int)((int64_t)spare * len(cur[i]) / tot);
            used += P[i];
        }
        for (int i = 0; used < sms; i = (i + 1) % n, ++used) ++P[i];
        size_t off = 0;
        for (int i = 0; i < n; ++i) {
            Plan plan;
            if (!make_plan(q, len(cur[i]), P[i], ps, plan)) return false;
            w.plans.push_back(plan);
            w.offs.push_back(off);
            off += align_up(plan.total);
            w.smem = std::max(w.smem, plan.p.smem_bytes);
        }
        w.bytes = off;
        waves.push_back(std::move(w));
        cur.clear();
        tot = 0;
        need = 0;
        return true;
    };
    for (int b = 0; b < q.B; ++b) {
        if (len(b) == 0) continue;
        if (min_ctas(b) > sms) return false;
        if (!cur.empty() && (need + min_ctas(b) > sms || (int)cur.size() == kMaxWave))
            if (!flush()) return false;
        cur.push_back(b);
        tot += len(b);
        need += min_ctas(b);
    }
    return flush();
}

// Batches go in waves when every prompt of every wave has a plan.
bool use_waves(const ScoreProblem& q) { return q.B > 1; }

}  // namespace

unsigned long long score_tc_set_exchange_wait_ns(unsigned long long ns) {
    return g_exchange_wait_ns.exchange(ns == 0 ? kTimeoutNs : ns);
}


// The first pass has the most steps (the largest workspace).
Pass first_pass(const ScoreProblem& q) { return Pass{0, std::min(q.N, steps_per_pass(q))}; }

// The plan of one bf16 prompt of M tokens on `sms` SMs (first pass), for tests
// of the planner: out = {F, Pc, P, n_tiles_max, tiles_per_group, land, held,
// lag, smem_bytes}.  Returns false when the tensor-core path does not take it.
bool score_tc_plan_of(int L, int H, int H_kv, int d, int64_t M, int N, int sms, int out[9]) {
    ScoreProblem q{};
    q.B = 1; q.L = L; q.H = H; q.H_kv = H_kv; q.d = d; q.N = N;
    q.T = M; q.max_M = M; q.dtype = SP_BF16;
    if (H_kv < 1 || H % H_kv != 0 || !shape_ok(q)) return false;
    Plan plan;
    if (!make_plan(q, M, sms, first_pass(q), plan)) return false;
    const TcParams& p = plan.p;
    const int v[9] = {p.F, p.Pc, p.P, p.n_tiles_max, p.tiles_per_group, p.land, p.held, p.lag, p.smem_bytes};
    for (int i = 0; i < 9; ++i) out[i] = v[i];
    return true;
}

bool score_tc_supported(const ScoreProblem& q) {
    Plan plan;
    return shape_ok(q) && make_plan(q, q.max_M, sm_count_or(148), first_pass(q), plan);
}

size_t score_tc_ws_bytes(const ScoreProblem& q) {
    // prompt after prompt (and pass after pass) the workspace is reused: the
    // largest prompt of the first pass needs the most
    if (!shape_ok(q)) return 0;
    Plan plan;
    size_t bytes = make_plan(q, q.max_M, kMaxCtas, first_pass(q), plan) ? plan.total : 0;
    if (bytes > 0 && use_waves(q)) {
        std::vector<Wave> waves;
        if (plan_waves(q, sm_count_or(148), first_pass(q), waves))
            for (const Wave& w : waves) bytes = std::max(bytes, w.bytes);
    }
    return bytes;
}

// One prompt (b) of a packed batch: its plan, workspace pointers and launches.
static sp_status launch_prompt(const ScoreProblem& q, int b, bool first, const KMaps& maps, int sms, Pass ps,
                               void* ws, cudaStream_t st) {
    const int64_t M = q.cu_M_host[b + 1] - q.cu_M_host[b];
    Plan plan;
    if (!make_plan(q, M, sms, ps, plan)) {
        set_error("sp_score: prompt %d (%lld tokens) is outside the tensor-core path", b, (long long)M);
        return SP_EUNSUPPORTED;
    }
    uint8_t* w = static_cast<uint8_t*>(ws);
    bind_prompt(q, b, first, w, w, plan);
    const TcParams& p = plan.p;
    if (p.d == 64) tc_prep_kernel<1><<<p.S, 256, 0, st>>>(p);
    else tc_prep_kernel<2><<<p.S, 256, 0, st>>>(p);
    SP_LAUNCH_CHECK();
    switch (q.d * 32 + p.G) {
        case 64 * 32 + 1: return launch_kernel<64, 1>(maps, p, st);
        case 64 * 32 + 2: return launch_kernel<64, 2>(maps, p, st);
        case 64 * 32 + 4: return launch_kernel<64, 4>(maps, p, st);
        case 64 * 32 + 8: return launch_kernel<64, 8>(maps, p, st);
        case 64 * 32 + 16: return launch_kernel<64, 16>(maps, p, st);
        case 128 * 32 + 1: return launch_kernel<128, 1>(maps, p, st);
        case 128 * 32 + 2: return launch_kernel<128, 2>(maps, p, st);
        case 128 * 32 + 4: return launch_kernel<128, 4>(maps, p, st);
        case 128 * 32 + 8: return launch_kernel<128, 8>(maps, p, st);
        case 128 * 32 + 16: return launch_kernel<128, 16>(maps, p, st);
        default: break;
    }
    set_error("sp_score: no tensor-core kernel for d=%d G=%d", q.d, p.G);
    return SP_EUNSUPPORTED;
}

// One wave: one preparation launch and one cooperative launch for all its prompts.
static sp_status launch_wave(const ScoreProblem& q, Wave& wv, bool first, const KMaps& maps, void* ws,
                             cudaStream_t st) {
    static_assert(sizeof(TcBatch) < 32000, "a wave's parameters must fit the kernel parameter space");
    TcBatch bt;
    bt.nb = (int)wv.prompts.size();
    bt.cta0[0] = 0;
    uint8_t* w = static_cast<uint8_t*>(ws);
    for (int i = 0; i < bt.nb; ++i) {
        Plan& plan = wv.plans[i];
        bind_prompt(q, wv.prompts[i], first && i == 0, w, w + wv.offs[i], plan);
        bt.p[i] = plan.p;
        bt.cta0[i + 1] = bt.cta0[i] + plan.p.P;
    }
    if (bt.p[0].d == 64) tc_prep_batch_kernel<1><<<bt.nb * bt.p[0].S, 256, 0, st>>>(bt);
    else tc_prep_batch_kernel<2><<<bt.nb * bt.p[0].S, 256, 0, st>>>(bt);
    SP_LAUNCH_CHECK();
    switch (q.d * 32 + bt.p[0].G) {
        case 64 * 32 + 1: return launch_batch<64, 1>(maps, bt, wv.smem, st);
        case 64 * 32 + 2: return launch_batch<64, 2>(maps, bt, wv.smem, st);
        case 64 * 32 + 4: return launch_batch<64, 4>(maps, bt, wv.smem, st);
        case 64 * 32 + 8: return launch_batch<64, 8>(maps, bt, wv.smem, st);
        case 64 * 32 + 16: return launch_batch<64, 16>(maps, bt, wv.smem, st);
        case 128 * 32 + 1: return launch_batch<128, 1>(maps, bt, wv.smem, st);
        case 128 * 32 + 2: return launch_batch<128, 2>(maps, bt, wv.smem, st);
        case 128 * 32 + 4: return launch_batch<128, 4>(maps, bt, wv.smem, st);
        case 128 * 32 + 8: return launch_batch<128, 8>(maps, bt, wv.smem, st);
        case 128 * 32 + 16: return launch_batch<128, 16>(maps, bt, wv.smem, st);
        default: break;
    }
    set_error("sp_score: no tensor-core kernel for d=%d G=%d", q.d, bt.p[0].G);
    return SP_EUNSUPPORTED;
}

sp_status score_tc_launch(const ScoreProblem& q, void* ws, cudaStream_t st) {
    const int sms = sm_count_or(0);
    if (sms < 1 || !shape_ok(q)) {
        set_error("sp_score: shape outside the tensor-core path");
        return SP_EUNSUPPORTED;
    }
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) {
        set_error("sp_score: cuTensorMapEncodeTiled is unavailable from the driver");
        return SP_ECUDA;
    }
    const int S = q.L * q.H_kv;
    // K viewed as a 2D tensor of L*H_kv*T rows (T: the packed tokens) by d bf16 columns;
    // 64-column boxes of 128 rows (full tiles) and of 32 rows (ragged last tiles).
    KMaps maps;
    const cuuint64_t gdim[2] = {(cuuint64_t)q.d, (cuuint64_t)S * (cuuint64_t)q.T};
    const cuuint64_t gstride[1] = {(cuuint64_t)q.d * 2};
    const cuuint32_t estride[2] = {1u, 1u};
    for (int k = 0; k < 2; ++k) {
        const cuuint32_t box[2] = {64u, (cuuint32_t)(k == 0 ? kTileRows : kBoxRows)};
        const CUresult cr = enc(k == 0 ? &maps.full : &maps.tail, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                const_cast<void*>(q.K), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr != CUDA_SUCCESS) {
            set_error("sp_score: cuTensorMapEncodeTiled failed (%d)", (int)cr);
            return SP_ECUDA;
        }
    }

    // Pass after pass (steps j0 .. j0 + n - 1 each, stream-ordered, sharing
    // the workspace); the first launch of the call clears the status.
    const size_t ws_cap = score_tc_ws_bytes(q);
    const int per = steps_per_pass(q);
    bool first = true;
    for (int j0 = 0; j0 < q.N; j0 += per) {
        const Pass ps{j0, std::min(per, q.N - j0)};
        // a batch: wave after wave, each wave's prompts side by side on the SMs
        // (stream order separates the waves, which reuse the workspace)
        std::vector<Wave> waves;
        bool done = false;
        if (use_waves(q) && plan_waves(q, sms, ps, waves)) {
            size_t need = 0;
            for (const Wave& w : waves) need = std::max(need, w.bytes);
            if (need <= ws_cap) {
                for (Wave& w : waves) {
                    const sp_status s = launch_wave(q, w, first, maps, ws, st);
                    if (s != SP_OK) return s;
                    first = false;
                }
                done = true;
            }
        }
        if (done) continue;
        // otherwise one prompt after another, each with its own plan over all
        // SMs; they share the workspace (stream order separates them)
        for (int b = 0; b < q.B; ++b) {
            if (q.cu_M_host[b + 1] == q.cu_M_host[b]) continue;
            const sp_status s = launch_prompt(q, b, first, maps, sms, ps, ws, st);
            if (s != SP_OK) return s;
            first = false;
        }
    }
    return SP_OK;
}

}  // namespace sp
