// sample.cu -- k_sample: the emitted token of every sampling request.
//
// Residual ("深入推测解码" 保证原始分布 step 4; "投机采样" 第四步 and 第五步):
// at the first rejected row e the token is drawn from norm(max(0, p_e - q_e)).
// Bonus ("投机采样" output-length case 3): when all drafts are accepted one token
// is drawn from p_{n_b}.  Both draws are an inverse CDF with the row's emission
// uniform u' (Philox lane 1): the smallest x with C(x) >= u' * C(V-1), C the
// prefix sum of the weights in token order.
//
// The CDF is evaluated in two levels so that only one chunk is ever scanned:
//   level 1: per-chunk masses (residual: computed here, CH2 tokens per CTA
//            unit; bonus: the row-stat partials of k_row_stats), prefix-summed
//            in float64 in chunk order -> the chunk c* holding u' * C(V-1);
//   level 2: the chunk c* is re-read, its weights recomputed with the same
//            float32 expression as level 1, block-scanned in float64, and the
//            first token whose running sum reaches the remaining mass is taken
//            (zero-mass tokens are never taken; if rounding leaves the
//            threshold beyond the chunk, its last token of positive mass is).
// Residual chunk sums of one request are spread over CTAs; the CTA that
// finishes the last one (atomic counter, threadfence pattern) runs level 2.
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace sv {

namespace {

constexpr int NW = SAMPLE_THREADS / 32;

struct Smem {
    double red[NW];
    int ired[NW];
    double t_level2;
    double mass;
    int chunk;
    int last;
};

__device__ __forceinline__ double block_sum(double v, Smem& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) sm.red[warp] = v;
    __syncthreads();
    double s = 0.0;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += sm.red[w];  // same order in every thread
    return s;
}

// Exclusive prefix (token order = thread order) of one double per thread.
__device__ __forceinline__ double block_excl_scan(double v, Smem& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    double incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) sm.red[warp] = incl;
    __syncthreads();
    double base = 0.0;
    for (int w = 0; w < warp; ++w) base += sm.red[w];
    return base + incl - v;
}

__device__ __forceinline__ int block_min_int(int v, Smem& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_min_int(v);
    __syncthreads();
    if (lane == 0) sm.ired[warp] = v;
    __syncthreads();
    int r = INT_MAX;
#pragma unroll
    for (int w = 0; w < NW; ++w) r = min(r, sm.ired[w]);
    return r;
}

__device__ __forceinline__ int block_max_int(int v, Smem& sm) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max_int(v);
    __syncthreads();
    if (lane == 0) sm.ired[warp] = v;
    __syncthreads();
    int r = INT_MIN;
#pragma unroll
    for (int w = 0; w < NW; ++w) r = max(r, sm.ired[w]);
    return r;
}

// max(0, p - q) with p = 2^((l - m) kappa) / Z; the same float32 operations
// at both levels so that a token's weight is bit-identical in both.
__device__ __forceinline__ float resid(float l, float q, float m, float kappa, float invZ) {
    const float p = __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(l, m), kappa)), invZ);
    return fmaxf(__fsub_rn(p, q), 0.f);
}

// 8 consecutive logits starting at element e (e % 8 == 0), read-only path.
template <int DT>
__device__ __forceinline__ void load8(const void* logits, size_t e, float (&f)[8]) {
    if constexpr (DT == SPEC_BF16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(
            reinterpret_cast<const uint16_t*>(logits) + e));
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else {
        const float4* p = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(logits) + e);
        const float4 a = __ldg(p), c = __ldg(p + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
    }
}
__device__ __forceinline__ void load8q(const float* q, size_t e, float (&f)[8]) {
    const float4* p = reinterpret_cast<const float4*>(q + e);
    const float4 a = __ldg(p), c = __ldg(p + 1);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
}

// Level 1 of the residual: mass of chunk c (CH2 tokens) of row rec.erow.
template <int DT>
__device__ double residual_chunk_sum(const Params& P, const ReqRec& rec, int c, Smem& sm) {
    const size_t lrow = ((size_t)rec.b * P.K1 + rec.erow) * P.V;
    const size_t qrow = ((size_t)rec.b * P.K + rec.erow) * P.V;
    const float invZ = float(1.0 / rec.Z);
    constexpr int G = CH2 / 8 / SAMPLE_THREADS;  // 8-token groups per thread
    float gs[G];
#pragma unroll
    for (int k = 0; k < G; ++k) {
        const int e0 = c * CH2 + (k * SAMPLE_THREADS + threadIdx.x) * 8;
        gs[k] = 0.f;
        if (e0 < P.V) {
            float l[8], q[8], r[8];
            load8<DT>(P.logits, lrow + e0, l);
            load8q(P.probs, qrow + e0, q);
#pragma unroll
            for (int e = 0; e < 8; ++e) r[e] = resid(l[e], q[e], rec.m, rec.kappa, invZ);
#pragma unroll
            for (int h = 4; h; h >>= 1)
#pragma unroll
                for (int e = 0; e < h; ++e) r[e] = __fadd_rn(r[e], r[e + h]);
            gs[k] = r[0];
        }
    }
#pragma unroll
    for (int h = G / 2; h; h >>= 1)
#pragma unroll
        for (int k = 0; k < h; ++k) gs[k] = __fadd_rn(gs[k], gs[k + h]);
    return block_sum(double(gs[0]), sm);
}

// Level 1 over `nc` chunk masses mass(c) (c in order): total S = last prefix,
// then the first chunk whose prefix reaches u * S.  Run by warp 0; results in sm.
template <typename MassFn>
__device__ void pick_chunk(int nc, float u, MassFn mass, Smem& sm) {
    const int lane = threadIdx.x & 31;
    if (threadIdx.x >= 32) return;
    double carry = 0.0;
    for (int c0 = 0; c0 < nc; c0 += 32) {
        double v = c0 + lane < nc ? mass(c0 + lane) : 0.0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
    const double S = carry;
    const double t = double(u) * S;
    int chosen = -1;
    double before = 0.0;
    carry = 0.0;
    for (int c0 = 0; c0 < nc && chosen < 0; c0 += 32) {
        const double m = c0 + lane < nc ? mass(c0 + lane) : 0.0;
        double v = m;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        const double incl = carry + v;
        const unsigned hit = __ballot_sync(0xffffffffu, c0 + lane < nc && incl >= t && m > 0.0);
        const double prev = __shfl_up_sync(0xffffffffu, incl, 1);
        if (hit) {
            const int l = __ffs(hit) - 1;
            chosen = c0 + l;
            before = __shfl_sync(0xffffffffu, lane == 0 ? carry : prev, l);
        }
        carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) {
        sm.mass = S;
        sm.chunk = chosen;
        sm.t_level2 = t - before;
    }
}

template <int DT>
__device__ void write_emit(const Params& P, const ReqRec& rec, int x, int mode, double mass) {
    P.out_ids[(size_t)rec.b * P.K1 + rec.erow] = x;
    if (P.dbg_req) {
        float* d = P.dbg_req + (size_t)rec.b * 4;
        d[0] = float(mode);
        d[1] = float(rec.erow);
        d[2] = float(mass);
        d[3] = rec.u2;
    }
}

// Draw from p of row rec.erow using the row-stat partials (bonus token, or the
// residual when it has no mass).
template <int DT>
__device__ void emit_from_p(const Params& P, const ReqRec& rec, int mode, Smem& sm) {
    const Partial* part = P.part + ((size_t)rec.b * P.K1 + rec.erow) * P.C;
    const float m = rec.m, kappa = rec.kappa;
    auto wmass = [&](int c) -> double {
        const Partial q = part[c];
        if (q.m == -INFINITY || q.z == 0.0) return 0.0;
        return q.z * exp2(double(__fmul_rn(__fsub_rn(q.m, m), kappa)));
    };
    pick_chunk(P.C, rec.u2, wmass, sm);
    __syncthreads();
    const int c = sm.chunk;
    const double S = sm.mass;
    if (c < 0) {  // no mass at all (cannot happen for a row with a finite logit)
        if (threadIdx.x == 0) write_emit<DT>(P, rec, 0, mode, S);
        __syncthreads();
        return;
    }
    const Partial pc = part[c];
    const double f_c = exp2(double(__fmul_rn(__fsub_rn(pc.m, m), kappa)));
    const double t = sm.t_level2 / f_c;  // remaining mass in the chunk's own scale
    // level 2: TILE tokens, TILE / SAMPLE_THREADS consecutive tokens per thread
    constexpr int PT = TILE / SAMPLE_THREADS;
    const size_t lrow = ((size_t)rec.b * P.K1 + rec.erow) * P.V;
    const int e0 = c * TILE + threadIdx.x * PT;
    float w[PT];
    double ts = 0.0;
#pragma unroll
    for (int k = 0; k < PT; k += 8) {
        float l[8];
        if (e0 + k < P.V) {
            load8<DT>(P.logits, lrow + e0 + k, l);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) l[e] = -INFINITY;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            w[k + e] = ex2_approx(__fmul_rn(__fsub_rn(l[e], pc.m), kappa));
            ts += double(w[k + e]);
        }
    }
    double acc = block_excl_scan(ts, sm);
    int cand = INT_MAX, lastpos = INT_MIN;
#pragma unroll
    for (int k = 0; k < PT; ++k) {
        acc += double(w[k]);
        if (w[k] > 0.f) {
            lastpos = e0 + k;
            if (cand == INT_MAX && acc >= t) cand = e0 + k;
        }
    }
    int x = block_min_int(cand, sm);
    if (x == INT_MAX) x = block_max_int(lastpos, sm);
    if (threadIdx.x == 0) write_emit<DT>(P, rec, x == INT_MIN ? c * TILE : x, mode, S);
    __syncthreads();
}

// Level 2 of the residual for queued request i (run by the CTA that finished
// its last chunk sum).
template <int DT>
__device__ void emit_residual(const Params& P, const ReqRec& rec, int i, Smem& sm) {
    const double* rs = P.rsum + (size_t)i * P.C2;
    pick_chunk(P.C2, rec.u2, [&](int c) -> double { return __ldcg(rs + c); }, sm);
    __syncthreads();
    const int c = sm.chunk;
    const double S = sm.mass;
    if (c < 0 || !(S > 0.0)) {  // residual without mass: draw from p instead
        __syncthreads();
        emit_from_p<DT>(P, rec, MODE_FALLBACK, sm);
        return;
    }
    const double t = sm.t_level2;
    const float invZ = float(1.0 / rec.Z);
    constexpr int PT = CH2 / SAMPLE_THREADS;  // consecutive tokens per thread
    const size_t lrow = ((size_t)rec.b * P.K1 + rec.erow) * P.V;
    const size_t qrow = ((size_t)rec.b * P.K + rec.erow) * P.V;
    const int e0 = c * CH2 + threadIdx.x * PT;
    float r[PT];
    double ts = 0.0;
#pragma unroll
    for (int k = 0; k < PT; k += 8) {
        if (e0 + k < P.V) {
            float l[8], q[8];
            load8<DT>(P.logits, lrow + e0 + k, l);
            load8q(P.probs, qrow + e0 + k, q);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                r[k + e] = resid(l[e], q[e], rec.m, rec.kappa, invZ);
                ts += double(r[k + e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) r[k + e] = 0.f;
        }
    }
    double acc = block_excl_scan(ts, sm);
    int cand = INT_MAX, lastpos = INT_MIN;
#pragma unroll
    for (int k = 0; k < PT; ++k) {
        acc += double(r[k]);
        if (r[k] > 0.f) {
            lastpos = e0 + k;
            if (cand == INT_MAX && acc >= t) cand = e0 + k;
        }
    }
    int x = block_min_int(cand, sm);
    if (x == INT_MAX) x = block_max_int(lastpos, sm);
    if (threadIdx.x == 0) write_emit<DT>(P, rec, x == INT_MIN ? c * CH2 : x, MODE_RESIDUAL, S);
    __syncthreads();
}

}  // namespace

template <int DT>
__device__ __forceinline__ void sample_body(const Params& P) {
    __shared__ Smem sm;
    griddep_launch_dependents();
    griddep_wait();  // decisions and queues of k_accept
    const int n_res = P.hdr[HDR_NRES], n_bonus = P.hdr[HDR_NBONUS];
    const long long res_units = (long long)n_res * P.C2;
    const long long units = res_units + n_bonus;
    for (long long unit = blockIdx.x; unit < units; unit += gridDim.x) {
        if (unit < res_units) {
            const int i = int(unit / P.C2), c = int(unit - (long long)i * P.C2);
            const ReqRec rec = P.reqs[P.res_list[i]];
            const double s = residual_chunk_sum<DT>(P, rec, c, sm);
            if (threadIdx.x == 0) {
                P.rsum[(size_t)i * P.C2 + c] = s;
                __threadfence();
                sm.last = (atomicAdd(&P.res_cnt[i], 1) == P.C2 - 1);
            }
            __syncthreads();
            const bool last = sm.last;
            __syncthreads();
            if (last) {
                __threadfence();
                emit_residual<DT>(P, rec, i, sm);
            }
        } else {
            const ReqRec rec = P.reqs[P.bonus_list[unit - res_units]];
            emit_from_p<DT>(P, rec, MODE_BONUS, sm);
        }
        __syncthreads();
    }
}

__global__ void __launch_bounds__(SAMPLE_THREADS) k_sample_f32(Params P) { sample_body<SPEC_F32>(P); }
__global__ void __launch_bounds__(SAMPLE_THREADS) k_sample_bf16(Params P) { sample_body<SPEC_BF16>(P); }

}  // namespace sv
