// draw.cuh -- the two-level inverse CDF of the emitted token.
//
// Residual ("深入推测解码" 保证原始分布 step 4; "投机采样" 第四步, 第五步): at
// the first rejected row e the token is drawn from norm(max(0, p_e - q_e)).
// Bonus ("投机采样" output-length case 3): with every draft accepted, one
// token is drawn from p_{n_b}.  Both draws take the smallest x with
// C(x) >= u' * C(V-1), C the prefix sum of the weights in token order, u' the
// row's emission uniform.  Level 1 picks the 2048-token chunk from per-chunk
// masses (float64 prefix in chunk order); level 2 scans that chunk's weights
// in token order.
#pragma once

#include <cfloat>
#include <climits>

#include "common.cuh"

namespace sv {

namespace {

template <int DT>
struct Stage {
    static constexpr int ESZ = DT == SPEC_BF16 ? 2 : 4;
    static constexpr int LB = TILE * ESZ;  // logits chunk
    static constexpr int QB = TILE * 4;    // draft-probability chunk
    static constexpr int BYTES = LB + QB;
};

// max(0, p - q) with p = 2^((l - m) kappa) / Z, written against the row's
// offset c = offset_of(m, kappa) like every other weight of the row; the same float32
// operations at both levels so that a token's weight is bit-identical in both.
__device__ __forceinline__ float resid(float l, float q, float m, float c, float kappa,
                                      float invZ) {
    const float p = __fmul_rn(ex2_approx(weight_arg(l, m, c, kappa)), invZ);
    return fmaxf(__fsub_rn(p, q), 0.f);
}

// The 8 logits of group g of a staged chunk.
template <int DT>
__device__ __forceinline__ void smem_logits8(const uint8_t* st, int g, float (&f)[8]) {
    if constexpr (DT == SPEC_BF16) {
        const uint4 v = reinterpret_cast<const uint4*>(st)[g];
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else {
        const float4 a = reinterpret_cast<const float4*>(st)[2 * g];
        const float4 c = reinterpret_cast<const float4*>(st)[2 * g + 1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
    }
}
__device__ __forceinline__ void smem_q8(const uint8_t* stq, int g, float (&f)[8]) {
    const float4 a = reinterpret_cast<const float4*>(stq)[2 * g];
    const float4 c = reinterpret_cast<const float4*>(stq)[2 * g + 1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
}


struct Pick {
    int chunk;      // chosen chunk, -1 if the total mass is not positive
    double before;  // mass of the chunks before it
    double total;   // total mass S (the last prefix)
};

__device__ __forceinline__ double warp_incl_scan(double x) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    return x;
}

// Level 1 over nc chunk masses mass(c) in chunk order, by one warp: S = the
// total; the chosen chunk is the first of positive mass whose prefix reaches
// u * S (the last of positive mass if rounding leaves u * S beyond every
// prefix).  Up to PICK_NB * 32 chunks are loaded at once (one round trip) and
// summed with one warp scan; beyond, block by block.
constexpr int PICK_NB = 4;

// Lane l holds chunks PICK_NB*l .. PICK_NB*l + PICK_NB - 1 (0 past nc), so
// chunk order runs lane by lane.  For nc <= PICK_NB * 32.
template <typename MassFn>
__device__ __forceinline__ void load_masses(int nc, MassFn mass, double (&v)[PICK_NB]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < PICK_NB; ++i) {
        const int c = lane * PICK_NB + i;
        v[i] = c < nc ? mass(c) : 0.0;
    }
}

// The pick over masses held as load_masses holds them: one warp scan of the
// lane sums, then a walk within the lane.
__device__ __forceinline__ Pick pick_loaded(float u, const double (&v)[PICK_NB]) {
    const int lane = threadIdx.x & 31;
    constexpr int NB = PICK_NB;
    Pick pk;
    pk.chunk = -1;
    pk.before = 0.0;
    {
        double sl = 0.0;
#pragma unroll
        for (int i = 0; i < NB; ++i) sl += v[i];
        const double incl = warp_incl_scan(sl);
        const double total = __shfl_sync(0xffffffffu, incl, 31);
        pk.total = total;
        if (!(total > 0.0)) return pk;
        const double t = double(u) * total;
        const double ex = __shfl_up_sync(0xffffffffu, incl, 1);
        double run = lane == 0 ? 0.0 : ex;
        int cand = -1, lastpos = -1;
        double cbefore = 0.0, lbefore = 0.0;
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const double nr = run + v[i];
            if (v[i] > 0.0) {
                if (cand < 0 && nr >= t) {
                    cand = lane * NB + i;
                    cbefore = run;
                }
                lastpos = lane * NB + i;
                lbefore = run;
            }
            run = nr;
        }
        unsigned hit = __ballot_sync(0xffffffffu, cand >= 0);
        if (hit) {
            const int l = __ffs(hit) - 1;
            pk.chunk = __shfl_sync(0xffffffffu, cand, l);
            pk.before = __shfl_sync(0xffffffffu, cbefore, l);
        } else {  // rounding left the threshold past the end: the last chunk of positive mass
            hit = __ballot_sync(0xffffffffu, lastpos >= 0);
            const int l = 31 - __clz(hit);
            pk.chunk = __shfl_sync(0xffffffffu, lastpos, l);
            pk.before = __shfl_sync(0xffffffffu, lbefore, l);
        }
        return pk;
    }
}

template <typename MassFn>
__device__ __forceinline__ Pick pick_chunk(int nc, float u, MassFn mass) {
    const int lane = threadIdx.x & 31;
    if (nc <= PICK_NB * 32) {
        double v[PICK_NB];
        load_masses(nc, mass, v);
        return pick_loaded(u, v);
    }
    Pick pk;
    pk.chunk = -1;
    pk.before = 0.0;
    double carry = 0.0;
    for (int c0 = 0; c0 < nc; c0 += 32)
        carry = carry + __shfl_sync(0xffffffffu,
                                    warp_incl_scan(c0 + lane < nc ? mass(c0 + lane) : 0.0), 31);
    pk.total = carry;
    if (!(carry > 0.0)) return pk;
    const double t = double(u) * carry;
    carry = 0.0;
    for (int c0 = 0; c0 < nc; c0 += 32) {
        const double m = c0 + lane < nc ? mass(c0 + lane) : 0.0;
        const double incl = carry + warp_incl_scan(m);
        const double prev = __shfl_up_sync(0xffffffffu, incl, 1);
        const unsigned hit = __ballot_sync(0xffffffffu, c0 + lane < nc && incl >= t && m > 0.0);
        if (hit) {
            const int l = __ffs(hit) - 1;
            pk.chunk = c0 + l;
            pk.before = __shfl_sync(0xffffffffu, lane == 0 ? carry : prev, l);
            break;
        }
        carry = __shfl_sync(0xffffffffu, incl, 31);
    }
    return pk;
}

// The reciprocal of d, an exact power of two of normal range, by its exponent
// bits (the product by it then rounds as the quotient would); any other d is
// divided as usual.
__device__ __forceinline__ double pow2_recip(double d) {
    const long long bits = __double_as_longlong(d);
    const long long e = (bits >> 52) & 0x7FF;
    if (e == 0 || e >= 2046 || (bits & 0xFFFFFFFFFFFFFLL) != 0) return 1.0 / d;
    return __longlong_as_double((2046LL - e) << 52);
}

// Level-2 sums are fixed point: a weight w (0 <= w <= 4 by construction:
// rebased token weights stay within 2^(+-1) of 1, residual weights are
// probabilities) counts as the integer nearest w 2^48, so the running sums of
// a chunk (2048 tokens, below 2^61) are exact integer additions: no float64
// arithmetic, whose rate is low on this GPU, and each weight is off by at
// most 2^-49.
__device__ __forceinline__ long long fx48(float w) {
    return w > 0.f ? __float2ll_rn(fminf(w, 4.f) * 0x1p48f) : 0LL;
}
// The level-2 target t in the same units: a running sum reaches t exactly
// when the integer sum reaches ceil(t 2^48).  NaN never is reached.
__device__ __forceinline__ long long fx48_target(double t) {
    const double s = ceil(t * 0x1p48);
    if (s != s || s >= 0x1p62) return 1LL << 62;
    return s > 0.0 ? (long long)s : 0LL;
}

// Level 2 over a staged chunk of nel tokens starting at token c0: weight8(g, w)
// gives the float32 weights of 8-token group g (same expression as level 1).
// Groups are visited in token order g = 32 k + lane; the running sums are the
// fixed-point sums above; returns the first token of positive weight whose
// running sum reaches t, or the chunk's last token of positive weight.
template <typename WeightFn>
__device__ __forceinline__ int level2(int c0, int nel, double t, WeightFn weight8) {
    const int lane = threadIdx.x & 31;
    constexpr int G = TILE / 8 / 32;
    const long long T = fx48_target(t);
    // block k by block k: the group sums of the block, their scan (carried
    // from the blocks before), and a stop at the first block that reaches T
    long long carry = 0, before = 0;
    int found = -1, last = -1;  // last: the last token of positive weight seen
#pragma unroll 1
    for (int k = 0; k < G; ++k) {
        const int g = k * 32 + lane;
        long long gs = 0;
        bool pos = false;
        if (g * 8 < nel) {
            float w[8];
            weight8(g, w);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                gs += fx48(w[e]);
                if (w[e] > 0.f) {
                    last = g * 8 + e;
                    pos = true;
                }
            }
        }
        long long incl = gs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        incl += carry;
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= T && pos);
        if (hit) {
            const int l = __ffs(hit) - 1;
            found = k * 32 + l;
            before = __shfl_sync(0xffffffffu, incl - gs, l);
            break;
        }
        carry = __shfl_sync(0xffffffffu, incl, 31);
    }
    int x = -1;
    if (found >= 0) {
        if (lane == (found & 31)) {  // the owning lane walks its group
            float w[8];
            weight8(found, w);
            long long run = before;
            int lastpos = -1;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                run += fx48(w[e]);
                if (w[e] > 0.f) {
                    lastpos = found * 8 + e;
                    if (x < 0 && run >= T) x = found * 8 + e;
                }
            }
            if (x < 0) x = lastpos;
        }
        x = __shfl_sync(0xffffffffu, x, found & 31);
    } else {
        x = warp_max_int(last);
    }
    return c0 + (x < 0 ? 0 : x);
}

}  // namespace

}  // namespace sv
