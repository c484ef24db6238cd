// row_stats.cu -- k_row_stats: the single pass over every target-logit row the
// verifier needs.
//
// For a sampling request the acceptance test needs p_j(x_j) =
// exp(l_j(x_j)/T - M_j) / Z_j (pages: "深入推测解码" 保证原始分布 step 3,
// "RTP-LLM Speculative Engine" 拒绝采样算法), so every element of row j enters
// the normaliser Z_j; a greedy request needs the argmax of the row
// ("投机采样" 验收标准 / 精确匹配).  Both are reductions over the vocabulary and
// the kernel streams each row from HBM exactly once.
//
// Work split: the compacted rows are cut into 2048-token chunks; the
// (row, chunk) tiles are divided into equal contiguous ranges, one per warp.
// Each warp runs its own STATS_STAGES-deep pipeline: lane 0 issues a 1-D bulk
// copy (cp.async.bulk, completion on a per-stage mbarrier) for the tile
// STATS_STAGES ahead while the warp reduces the current tile from shared
// memory with 16-byte loads: chunk max by warp shuffles, then the sum of
// exp2((l - max) * log2(e)/T) per lane in float32, summed across lanes in
// float64.  No block-wide barrier is used.  Output: one Partial per tile.
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace sv {

namespace {

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

}  // namespace

template <int DT>
__device__ __forceinline__ void row_stats_body(const Params& P) {
    using TL = Tile<DT>;
    constexpr int EPV = TL::EPV, VPL = TL::VPL;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[STATS_WARPS][STATS_STAGES];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* buf = smem + size_t(warp) * STATS_STAGES * TL::BYTES;
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < STATS_STAGES; ++s) mbar_init(&bars[warp][s], 1);
        fence_mbarrier_init();
    }
    __syncwarp();
    griddep_launch_dependents();
    griddep_wait();  // the row list of k_plan

    const long long R = P.hdr[HDR_ROWS];
    const long long T = R * P.C;
    const long long W = (long long)gridDim.x * STATS_WARPS;
    const long long w = (long long)blockIdx.x * STATS_WARPS + warp;
    const long long t0 = T * w / W, t1 = T * (w + 1) / W;
    if (t0 >= t1) return;

    // lane 0: issue tile t into stage s (row cache: consecutive tiles share rows)
    long long prow = -1;
    int pslot = 0;
    auto issue = [&](long long t, int s) {
        const long long r = t / P.C;
        const int c = int(t - r * P.C);
        if (r != prow) {
            prow = r;
            pslot = P.rowlist[r];
        }
        const int nel = min(TILE, P.V - c * TILE);
        const uint32_t bytes = uint32_t(nel) * TL::ESZ;
        const char* src = reinterpret_cast<const char*>(P.logits) +
                          ((size_t)pslot * P.V + (size_t)c * TILE) * TL::ESZ;
        mbar_arrive_expect_tx(&bars[warp][s], bytes);
        bulk_g2s(buf + s * TL::BYTES, src, bytes, &bars[warp][s]);
    };
    if (lane == 0) {
        for (int k = 0; k < STATS_STAGES && t0 + k < t1; ++k) issue(t0 + k, k);
    }

    long long crow = -1;
    int slot = 0;
    bool greedy = false;
    float kappa = 0.f;
    long long t = t0;
    bool timed_out = false;
    for (; t < t1; ++t) {
        const long long i = t - t0;
        const int s = int(i % STATS_STAGES);
        const uint32_t parity = uint32_t((i / STATS_STAGES) & 1);
        const long long r = t / P.C;
        const int c = int(t - r * P.C);
        if (r != crow) {
            crow = r;
            slot = P.rowlist[r];
            const float Tb = P.temp[slot / P.K1];
            greedy = (Tb == 0.f);
            kappa = greedy ? 0.f : kappa_of(Tb);
        }
        const int nvec = min(TILE, P.V - c * TILE) / EPV;

        const bool landed = mbar_wait_bounded(&bars[warp][s], parity);
        if (!__all_sync(0xffffffffu, landed)) {  // warp-uniform exit
            timed_out = true;
            break;
        }
        const uint4* v4 = reinterpret_cast<const uint4*>(buf + s * TL::BYTES);
        uint4 d[VPL];
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int v = k * 32 + lane;
            d[k] = v < nvec ? v4[v]
                            : make_uint4(TL::NEG_INF_WORD, TL::NEG_INF_WORD, TL::NEG_INF_WORD,
                                         TL::NEG_INF_WORD);
        }
        __syncwarp();  // every lane holds its share: the stage can be refilled
        if (lane == 0 && t + STATS_STAGES < t1) {
            fence_proxy_async_smem();
            issue(t + STATS_STAGES, s);
        }

        const int tok0 = c * TILE;
        Partial out;
        if (greedy) {
            // lowest index of the maximum: lanes visit their tokens in increasing order
            float best = -INFINITY;
            int bidx = INT_MAX;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                if (k * 32 + lane < nvec) {
                    float f[EPV];
                    unpack<DT>(d[k], f);
#pragma unroll
                    for (int e = 0; e < EPV; ++e) {
                        if (f[e] > best || bidx == INT_MAX) {
                            best = f[e];
                            bidx = tok0 + (k * 32 + lane) * EPV + e;
                        }
                    }
                }
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const float ob = __shfl_xor_sync(0xffffffffu, best, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
                if (ob > best || (ob == best && oi < bidx)) {
                    best = ob;
                    bidx = oi;
                }
            }
            out.m = best;
            out.amax = bidx;
            out.z = 0.0;
        } else {
            float lmax = -INFINITY;
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                float f[EPV];
                unpack<DT>(d[k], f);
#pragma unroll
                for (int e = 0; e < EPV; ++e) lmax = fmaxf(lmax, f[e]);
            }
            const float m = warp_max(lmax);
            double z = 0.0;
            if (m != -INFINITY) {
                float zs[VPL];
#pragma unroll
                for (int k = 0; k < VPL; ++k) {
                    float f[EPV];
                    unpack<DT>(d[k], f);
                    float e4[EPV];
#pragma unroll
                    for (int e = 0; e < EPV; ++e)
                        e4[e] = ex2_approx(__fmul_rn(__fsub_rn(f[e], m), kappa));
                    // pairwise within the vector
#pragma unroll
                    for (int h = EPV / 2; h; h >>= 1)
#pragma unroll
                        for (int e = 0; e < h; ++e) e4[e] = __fadd_rn(e4[e], e4[e + h]);
                    zs[k] = e4[0];
                }
#pragma unroll
                for (int h = VPL / 2; h; h >>= 1)
#pragma unroll
                    for (int k = 0; k < h; ++k) zs[k] = __fadd_rn(zs[k], zs[k + h]);
                z = warp_sum(double(zs[0]));
            }
            out.m = m;
            out.amax = -1;
            out.z = z;
        }
        if (lane == 0) P.part[(size_t)slot * P.C + c] = out;
    }

    if (timed_out) {
        if (lane == 0) atomicOr(P.status, int(SPEC_BADBIT_TIMEOUT));
        // let the copies still in flight land before the CTA's shared memory is released
        for (long long u = t; u < t1 && u < t + STATS_STAGES; ++u) {
            const long long i = u - t0;
            mbar_wait_bounded(&bars[warp][int(i % STATS_STAGES)],
                              uint32_t((i / STATS_STAGES) & 1), 100000000ull);
        }
    }
}

__global__ void __launch_bounds__(STATS_WARPS * 32) k_row_stats_f32(Params P) {
    row_stats_body<SPEC_F32>(P);
}
__global__ void __launch_bounds__(STATS_WARPS * 32) k_row_stats_bf16(Params P) {
    row_stats_body<SPEC_BF16>(P);
}

}  // namespace sv
