// common.cuh -- shared definitions of the spec_verify kernels (sm_103a).
//
// Pipeline of one spec_verify call (all on the caller's stream):
//   k_plan       1 CTA: validate num_draft / temperature (bad requests get
//                their -1 outputs here), compact the rows every request needs
//                (j = 0..n_b) into a row list, zero the counters.
//   k_row_stats  persistent, one independent bulk-copy pipeline per warp: for
//                every (valid row, 2048-token chunk) the chunk max, the sum of
//                exp2((l - max) * log2(e) / T) and (greedy rows) the argmax,
//                and the gathers l(x_j), q(x_j).  The all-rows pass is
//                balanced across SMs (each warp's last eighth is claimed by
//                whichever warp runs out first); an early-exit pass runs the
//                acceptance of each request it completes (accept.cuh).
//   k_accept_all one CTA per request (accept.cuh): merge the chunk partials
//                into per-row (max, Z, argmax), Philox uniforms, acceptance
//                bits, first-reject scan (ballot), write the accepted prefix,
//                queue sampling requests.
//   k_sample     persistent, warp pairs: the residual chunk masses of the
//                first rejected row of every rejecting request (streaming).
//   k_emit       one warp per queue slot: residual tokens (two-level inverse
//                CDF over the chunk masses) and bonus tokens (over the
//                row-stat partials).
// Every kernel executes griddepcontrol.wait before it touches its
// predecessor's output, so programmatic dependent launch (a build option,
// off by default: it measured no faster) is safe on any of the launches.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

// ---------------------------------------------------------------- sizes

// Launch-shape parameters (overridable at build time for tuning sweeps).
#ifndef SV_STATS_WARPS
#define SV_STATS_WARPS 8
#endif
#ifndef SV_STATS_STAGES
#define SV_STATS_STAGES 3
#endif
#ifndef SV_EMIT_WARPS
#define SV_EMIT_WARPS 1
#endif
#ifndef SV_SAMPLE_PAIRS
#define SV_SAMPLE_PAIRS 4
#endif
#ifndef SV_SAMPLE_STAGES
#define SV_SAMPLE_STAGES 2
#endif

constexpr int TILE = 2048;                    // tokens per row-stat chunk (one warp tile)
constexpr int STATS_WARPS = SV_STATS_WARPS;   // warps per k_row_stats CTA
constexpr int STATS_STAGES = SV_STATS_STAGES; // bulk-copy stages per warp
constexpr int EMIT_WARPS = SV_EMIT_WARPS;      // warps per k_emit CTA (1 staging buffer each)
constexpr int SAMPLE_PAIRS = SV_SAMPLE_PAIRS;    // warp pairs per k_sample CTA
constexpr int SAMPLE_STAGES = SV_SAMPLE_STAGES;  // staging buffers per k_sample warp pair
static_assert(SAMPLE_STAGES >= 2 && SAMPLE_PAIRS * SAMPLE_STAGES <= 32, "k_sample staging");
constexpr int PLAN_THREADS = 1024;

// HDR_ROUND + r: rows of early-exit round r (r >= 1), listed at rowlist + r * B
// HDR_CLAIM: tail segments claimed so far in the all-rows pass of k_row_stats
// HDR_VCLAIM: requests claimed so far by k_verify's CTAs
enum { HDR_ROWS = 0, HDR_NRES = 1, HDR_NBONUS = 2, HDR_STATUS = 3, HDR_CLAIM = 4, HDR_VCLAIM = 5,
       HDR_ROUND = 8, HDR_INTS = 64 };
static_assert(HDR_ROUND + SPEC_MAX_K + 1 <= HDR_INTS, "round counters overflow the header");
enum { MODE_BAD = -1, MODE_GREEDY = 0, MODE_RESIDUAL = 1, MODE_BONUS = 2, MODE_FALLBACK = 3,
       MODE_TYPICAL = 4 };
// acceptance rule of a call: the lossless test u <= p / q, or typical
// acceptance (p >= a hard threshold, no draft distribution)
enum { RULE_LOSSLESS = 0, RULE_TYPICAL = 1 };

// Per (row, chunk) statistics written by k_row_stats.
struct __align__(16) Partial {
    float m;     // max of the raw logits in the chunk (-inf if none finite)
    int amax;    // greedy rows: lowest token index attaining m; else -1
    double z;    // sampling rows: sum exp2((l - m) * kappa) over the chunk
};

// A queued sampling draw, written by the acceptance step.
struct __align__(16) ReqRec {
    int mode;     // MODE_*
    int erow;     // row the emitted token is drawn from
    float m;      // max of the raw logits of row erow
    float kappa;  // log2(e) / T (clamped to FLT_MAX)
    double Z;     // sum_x exp2((l(x) - m) * kappa) over row erow
    float u2;     // emission uniform of row erow (Philox lane 1)
    int b;        // request index
};

struct Params {
    const void* logits;
    const float* probs;
    const int32_t* ids;
    const int32_t* num_draft;
    const float* temp;
    int32_t* out_ids;
    int32_t* out_nacc;
    float* dbg_rows;
    float* dbg_req;
    int32_t* status;  // device status word (bits SPEC_BADBIT_*)
    // workspace sections
    int* hdr;
    int* rowlist;     // [B*(K+1)] slot = b*(K+1)+j of each compacted row
    int* req_flags;   // [B] bad bits found by k_plan
    Partial* part;    // [B*(K+1)*C]
    ReqRec* res_rec;    // [B] queued residual draws (queue order)
    ReqRec* bonus_rec;  // [B] queued bonus draws (queue order)
    float* rsum;      // [B*C] residual chunk sums (TILE-token chunks)
    float2* gath;     // [B*(K+1)] {l_j(x_j), q_j(x_j)} gathered by k_row_stats
    int* cnt;         // [B] (row, chunk) tiles of each request finished so far
    // early exit (round >= 0): this pass verifies row `round` of the requests
    // that accepted drafts 0..round-1; acceptance appends each survivor's next
    // row to the list of round + 1.  round = -1: every row in one pass.
    int round;
    // token-tree verification (tree != 0): row v of request b is node v, row c
    // of probs the draft distribution of node c; parents[b * K1 + c] < c
    int tree;
    const int32_t* parents;  // [B, N] (N = K1)
    int32_t* out_last;       // [B] last accepted node
    float* tmass;            // [B, C] per-chunk masses of a tree walk's residual
    uint64_t seed;
    const uint64_t* seed_dev;  // if set, the seed is read here when the kernels run
    uint32_t req_off;
    int rule;         // RULE_*
    float threshold;  // typical acceptance: keep x_j iff p_j(x_j) >= threshold
    int dtype;  // SPEC_F32 / SPEC_BF16
    int B, K, K1, V;
    int C;   // ceil(V / TILE): chunks per row
};

// Workspace layout (byte offsets, each section 256-byte aligned).
struct Layout {
    size_t hdr, rowlist, req_flags, part, res_rec, bonus_rec, rsum, gath, cnt, tmass, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline Layout make_layout(int B, int K, int V) {
    Layout L;
    const size_t K1 = size_t(K) + 1, C = (size_t(V) + TILE - 1) / TILE;
    size_t o = 0;
    L.hdr = o;        o = align256(o + HDR_INTS * sizeof(int));
    L.rowlist = o;    o = align256(o + size_t(B) * K1 * sizeof(int));
    L.req_flags = o;  o = align256(o + size_t(B) * sizeof(int));
    L.part = o;       o = align256(o + size_t(B) * K1 * C * sizeof(Partial));
    L.res_rec = o;    o = align256(o + size_t(B) * sizeof(ReqRec));
    L.bonus_rec = o;  o = align256(o + size_t(B) * sizeof(ReqRec));
    L.rsum = o;       o = align256(o + size_t(B) * C * sizeof(float));
    L.gath = o;       o = align256(o + size_t(B) * K1 * sizeof(float2));
    L.cnt = o;        o = align256(o + size_t(B) * sizeof(int));
    L.tmass = o;      o = align256(o + size_t(B) * C * sizeof(float));
    L.total = o;
    return L;
}

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbarrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase: false if it did not complete within
// `limit_ns` (the caller then reports SPEC_BADBIT_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// 2^x on the SFU (relative error a few ulp; 0 for x = -inf).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Token weights are w(x) = 2^((l(x) - m) kappa) for a reference maximum m.
// With the integer offset c = rint(RN(m * kappa)) the exponent is one FFMA,
// l * kappa - c (the product is exact inside the FMA); every weight of that
// reference then carries the common factor 2^(m kappa - c), which cancels in
// every normalised quantity.  The factor stays within 2^(+-1) while
// |c| < 2^24 (RN(m kappa) is then within 1/2 of m kappa, and c within 1/2 of
// that); for larger |c| (very small T, or very large logits) it would overflow
// or vanish, so the two-operation form (l - m) * kappa, with no factor, is
// used instead.  Both forms give about 2^0 at l == m and 0 far below it.
// Because offsets are integers, moving a sum from one reference to another is
// multiplying it by an exact power of two (rebase_factor).
constexpr float OFFSET_LIMIT = 16777216.f;  // 2^24
__device__ __forceinline__ float offset_of(float m, float kappa) {
    return rintf(__fmul_rn(m, kappa));
}
__device__ __forceinline__ bool offset_ok(float c) { return fabsf(c) < OFFSET_LIMIT; }
__device__ __forceinline__ float weight_arg(float l, float m, float c, float kappa) {
    return offset_ok(c) ? fmaf(l, kappa, -c) : __fmul_rn(__fsub_rn(l, m), kappa);
}
// Exponent of the factor that rebases weights computed against m_c onto m,
// each reference with or without its offset as offset_ok decides: the exact
// (m_c - m) kappa, less the factor 2^(m_c kappa - c_c) the weights of m_c
// carry, plus the factor 2^(m kappa - c_m) those of m carry (both exact by
// FMA).  With both offsets this is the integer c_c - c_m.
__device__ __forceinline__ float rebase_arg(float m_c, float m, float kappa) {
    const float cc = offset_of(m_c, kappa), cm = offset_of(m, kappa);
    const bool okc = offset_ok(cc), okm = offset_ok(cm);
    if (okc && okm) return __fsub_rn(cc, cm);
    float r = __fmul_rn(__fsub_rn(m_c, m), kappa);
    if (okc) r = __fsub_rn(r, fmaf(m_c, kappa, -cc));
    if (okm) r = __fadd_rn(r, fmaf(m, kappa, -cm));
    return r;
}
// 2^rebase_arg(m_c, m, kappa): with both offsets an exact power of two
// (integer exponent, scaled in integer arithmetic), otherwise exp2f of the
// mixed exponent.
__device__ __forceinline__ float rebase_factor(float m_c, float m, float kappa) {
    const float cc = offset_of(m_c, kappa), cm = offset_of(m, kappa);
    if (offset_ok(cc) && offset_ok(cm)) return scalbnf(1.f, int(cc) - int(cm));
    return exp2f(rebase_arg(m_c, m, kappa));
}

// Packed bf16x2 maximum (NaN operands lose).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two float32 lanes in one 64-bit register for the packed sm_100-family
// arithmetic (fma/add/mul/sub .rn.f32x2): each lane is rounded exactly as the
// scalar instruction rounds it, so packed and scalar sums agree bit for bit
// when they add in the same order.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// Sum of 8 floats in the order of the tree ((f0+f4)+(f2+f6)) + ((f1+f5)+(f3+f7)):
// two packed adds, one packed add, one scalar add.
__device__ __forceinline__ float sum8_tree(const float (&f)[8]) {
    const uint64_t s = f2_add(f2_add(f2_pack(f[0], f[1]), f2_pack(f[4], f[5])),
                              f2_add(f2_pack(f[2], f[3]), f2_pack(f[6], f[7])));
    float a, b;
    f2_unpack(s, a, b);
    return __fadd_rn(a, b);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// log2(e) / T, clamped so that (l - m) * kappa stays 0 at l == m.
__device__ __forceinline__ float kappa_of(float T) {
    const float k = 1.4426950408889634f / T;
    return k < 3.4028234663852886e38f ? k : 3.4028234663852886e38f;
}

// One logit as float (bf16 is the top half of an f32).
__device__ __forceinline__ float load_logit(const void* logits, int dtype, size_t idx) {
    if (dtype == SPEC_BF16) {
        const uint16_t h = __ldg(reinterpret_cast<const unsigned short*>(logits) + idx);
        return __uint_as_float(uint32_t(h) << 16);
    }
    return __ldg(reinterpret_cast<const float*>(logits) + idx);
}

// ---------------------------------------------------------------- Philox4x32-10
// J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel Random Numbers: As Easy as
// 1, 2, 3" (SC'11): ten rounds of two 32x32->64 multiplies with the key bumped
// by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}
// 32 random bits -> (0, 1]: ((x >> 8) + 1) * 2^-24 (exact in float).
__device__ __forceinline__ float uniform01(uint32_t x) {
    return float((x >> 8) + 1u) * 5.9604644775390625e-8f;
}
// Uniforms of row j of request b (global index b + req_off).
__device__ __forceinline__ uint4 row_block(const Params& P, int b, int j) {
    const uint64_t seed = P.seed_dev ? __ldg(reinterpret_cast<const unsigned long long*>(P.seed_dev))
                                     : P.seed;
    return philox4x32_10(make_uint4(uint32_t(b) + P.req_off, uint32_t(j), 0u, 0u),
                         uint32_t(seed), uint32_t(seed >> 32));
}

// ---------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// Single-instruction warp reductions (sm_100 family): max of f32 (NaN inputs
// ignored) and min of s32 over all 32 lanes.
__device__ __forceinline__ float redux_max_f32(float v) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ int redux_min_s32(int v) {
    int r;
    asm volatile("redux.sync.min.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
    return r;
}

__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ int warp_max_int(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Kernel entry points (defined in the .cu files).
__global__ void k_plan(Params P);
// host_io.cu: copies of spec_verify_host from mapped page-locked host memory
constexpr int HOST_IO_THREADS = 256;
__global__ void k_rows_in(const void* src, void* dst, const int32_t* num, int B, int K,
                          size_t row_bytes);
__global__ void k_qx_in(const float* src, float* dst, const int32_t* ids, const int32_t* num,
                        int B, int K, int V);
__global__ void k_qrows_in(Params P, const float* src);
__global__ void k_row_stats_f32(Params P);
__global__ void k_row_stats_bf16(Params P);
__global__ void k_sample_f32(Params P);
__global__ void k_sample_bf16(Params P);
__global__ void k_emit_f32(Params P);
__global__ void k_emit_bf16(Params P);

__global__ void k_accept_all(Params P);  // one CTA per request, after the row statistics
constexpr int ACCEPT_WARPS = 8;          // warps of a k_accept_all CTA
__global__ void k_tree_walk_f32(Params P);
__global__ void k_tree_walk_bf16(Params P);
#ifndef SV_TREE_THREADS
#define SV_TREE_THREADS 512
#endif
constexpr int TREE_THREADS = SV_TREE_THREADS;
constexpr int TREE_MAX_NODES = 32;

// verify.cu: the request-by-request verifier (one persistent CTA per SM)
constexpr int VCMAX = 96;  // longest row it takes, in 2048-token tiles (V <= 196608)
__global__ void k_prep(Params P);
__global__ void k_verify_bf16(Params P);
__global__ void k_verify_f32(Params P);
size_t verify_smem(int dtype);
int verify_threads(int dtype);

__global__ void k_philox_fill(uint64_t seed, const uint32_t* ctrs, int64_t n, uint32_t* out);

// Logits produced on the tensor cores from the target's hidden states
// (lmhead.cu): the rows k_plan listed are gathered into hid_c [rows, H], then
// one tcgen05 GEMM writes their bf16 logits and, in its epilogue, the
// row-statistics partials, the draft gathers and the acceptances.
struct LmHeadIn {
    const void* hidden;   // [B*(K+1), H] bf16
    const void* lm_head;  // [V, H] bf16
    int H;
    void* hid_c;          // workspace: [B*(K+1), H] bf16, the listed rows in list order
};
spec_status launch_lmhead_fused(const Params& P, const LmHeadIn& in, cudaStream_t st);

}  // namespace sv
