// stats.cuh -- the statistics of one staged 2048-token tile of a logits row
// (the unit of every streaming pass over the target's logits).
//
// A row's normaliser Z = sum_x 2^((l(x) - m) log2(e) / T) and, for greedy
// rows, its argmax are reductions over the whole vocabulary ("深入推测解码"
// 保证原始分布 step 3; "投机采样" 验收标准 / 精确匹配); a tile's share is one
// Partial {max, argmax, sum of weights against the tile's own offset}, and
// the consumers merge the tiles of a row (accept.cuh).
#pragma once

#include <climits>

#include "common.cuh"

namespace sv {

template <int DT>
struct Tile {
    static constexpr int ESZ = DT == SPEC_BF16 ? 2 : 4;   // bytes per logit
    static constexpr int EPV = 16 / ESZ;                  // logits per 16-byte vector
    static constexpr int BYTES = TILE * ESZ;              // one stage
    static constexpr int VPL = TILE / EPV / 32;           // vectors per lane
    static constexpr uint32_t NEG_INF_WORD = DT == SPEC_BF16 ? 0xFF80FF80u : 0xFF800000u;
};

template <int DT>
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[Tile<DT>::EPV]) {
    if constexpr (DT == SPEC_BF16) {
        f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
        f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
        f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
        f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
    } else {
        f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
    }
}

// Maximum of a lane's VPL vectors (tree; packed bf16x2 for bf16).
template <int DT>
__device__ __forceinline__ float lane_max(const uint4 (&d)[Tile<DT>::VPL]) {
    constexpr int VPL = Tile<DT>::VPL;
    if constexpr (DT == SPEC_BF16) {
        uint32_t w[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k) w[k] = bmax2(bmax2(d[k].x, d[k].y), bmax2(d[k].z, d[k].w));
#pragma unroll
        for (int h = VPL / 2; h; h >>= 1)
#pragma unroll
            for (int k = 0; k < h; ++k) w[k] = bmax2(w[k], w[k + h]);
        return fmaxf(bf16_lo(w[0]), bf16_hi(w[0]));
    } else {
        float w[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k)
            w[k] = fmaxf(fmaxf(__uint_as_float(d[k].x), __uint_as_float(d[k].y)),
                         fmaxf(__uint_as_float(d[k].z), __uint_as_float(d[k].w)));
#pragma unroll
        for (int h = VPL / 2; h; h >>= 1)
#pragma unroll
            for (int k = 0; k < h; ++k) w[k] = fmaxf(w[k], w[k + h]);
        return w[0];
    }
}


// The statistics of one staged tile (d: this lane's VPL vectors, nvec valid
// vectors, tok0 the tile's first token): greedy rows the tile max and the
// lowest index attaining it; sampling rows the tile max and the sum of
// 2^(l kappa - c) against the tile max's offset c (see weight_arg).
template <int DT>
__device__ __forceinline__ Partial tile_partial(const uint4 (&d)[Tile<DT>::VPL], int nvec, int tok0,
                                                bool greedy, float kappa) {
    constexpr int EPV = Tile<DT>::EPV, VPL = Tile<DT>::VPL;
    const int lane = threadIdx.x & 31;
    const float lmax = lane_max<DT>(d);
    Partial out;
    if (greedy) {
        // lowest index attaining the tile max: visiting tokens from high to
        // low index leaves the lowest hit
        const float m = redux_max_f32(lmax);
        int bidx = INT_MAX;
#pragma unroll
        for (int k = VPL - 1; k >= 0; --k) {
            if (k * 32 + lane < nvec) {
                float f[EPV];
                unpack<DT>(d[k], f);
#pragma unroll
                for (int e = EPV - 1; e >= 0; --e)
                    if (f[e] == m) bidx = tok0 + (k * 32 + lane) * EPV + e;
            }
        }
        out.m = m;
        out.amax = redux_min_s32(bidx);
        out.z = 0.0;
    } else {
        // each lane sums against its own maximum, so the ex2 loop does not
        // wait for the warp-wide maximum; one rescale per lane follows
        float zl = 0.f;
        if (lmax != -INFINITY) {
            const float cl = offset_of(lmax, kappa);
            float zs[VPL];
            if (offset_ok(cl)) {  // one FFMA + ex2 per token, FFMAs and adds in pairs
                const uint64_t kk = f2_pack(kappa, kappa), nc = f2_pack(-cl, -cl);
#pragma unroll
                for (int k = 0; k < VPL; ++k) {
                    float f[EPV];
                    unpack<DT>(d[k], f);
#pragma unroll
                    for (int e = 0; e < EPV; e += 2) {
                        f2_unpack(f2_fma(f2_pack(f[e], f[e + 1]), kk, nc), f[e], f[e + 1]);
                        f[e] = ex2_approx(f[e]);
                        f[e + 1] = ex2_approx(f[e + 1]);
                    }
                    if constexpr (EPV == 8) {
                        zs[k] = sum8_tree(f);
                    } else {
                        float a, b;
                        f2_unpack(f2_add(f2_pack(f[0], f[1]), f2_pack(f[2], f[3])), a, b);
                        zs[k] = __fadd_rn(a, b);
                    }
                }
            } else {  // offset too large (very small T): (l - max) * kappa
#pragma unroll
                for (int k = 0; k < VPL; ++k) {
                    float f[EPV];
                    unpack<DT>(d[k], f);
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        f[e] = ex2_approx(__fmul_rn(__fsub_rn(f[e], lmax), kappa));
#pragma unroll
                    for (int h = EPV / 2; h; h >>= 1)
#pragma unroll
                        for (int e = 0; e < h; ++e) f[e] = __fadd_rn(f[e], f[e + h]);
                    zs[k] = f[0];
                }
            }
#pragma unroll
            for (int h = VPL / 2; h > 1; h >>= 1)  // the same tree, two sums per add
#pragma unroll
                for (int k = 0; k < h; k += 2)
                    f2_unpack(f2_add(f2_pack(zs[k], zs[k + 1]), f2_pack(zs[k + h], zs[k + h + 1])),
                              zs[k], zs[k + 1]);
            zl = __fadd_rn(zs[0], zs[1]);
        }
        const float m = redux_max_f32(lmax);
        if (zl != 0.f) zl = __fmul_rn(zl, rebase_factor(lmax, m, kappa));
        out.m = m;
        out.amax = -1;
        out.z = double(warp_sum_f(zl));
    }
    return out;
}

}  // namespace sv
