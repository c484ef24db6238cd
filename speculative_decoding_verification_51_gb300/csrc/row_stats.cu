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
// (row, chunk) tiles are divided into equal contiguous ranges, one per warp
// (in the all-rows pass a warp streams the first 7/8 of its range and the
// last eighths go to whichever warps run out first: stream_balanced).
// Each warp runs its own STATS_STAGES-deep pipeline: lane 0 issues a 1-D bulk
// copy (cp.async.bulk, completion on a per-stage mbarrier) for the tile
// STATS_STAGES ahead while the warp reduces the current tile out of shared
// memory (16-byte loads, 64 tokens per lane):
//   sampling rows: each lane takes its maximum by a packed bf16x2 max tree and
//     sums 2^(l * kappa - c) against its own offset c = rint(max * kappa) (one
//     FFMA and one ex2 per token, pairwise float32 sums); the chunk maximum is
//     one redux.sync, each lane's sum is rebased onto it by an exact power of two, and the
//     lanes are summed by shuffles.  The stored sum is relative to the chunk's
//     offset rint(chunk max * kappa), as every consumer expects;
//   greedy rows: chunk max (redux), then the lowest index attaining it.
// While the tile holding the draft token x_j of a row is in shared memory its
// logit is copied out, and q_j(x_j) is fetched, for the acceptance test.
// No block-wide barrier and no float64 arithmetic (the FP64 pipe of this part
// is a small fraction of its FP32 rate).  Output: one Partial per tile.
//
// Acceptance: after the all-rows pass, k_accept_all (one CTA per request)
// runs every request's acceptance (accept_decide).  In an early-exit pass
// each warp adds the number of tiles it finished for a request to the
// request's counter (one atomic per contiguous run, after a threadfence) and
// the warp whose addition completes the row runs the acceptance at once, so
// that the survivors' next rows are listed before the next pass.  Nothing
// ever waits for another warp.
#include <cfloat>
#include <climits>

#include "accept.cuh"
#include "common.cuh"
#include "stats.cuh"

namespace sv {

namespace {

// Per-row facts a warp needs while it streams the row's chunks.
struct RowCtx {
    int slot;      // b * (K+1) + j
    int b;         // request
    int n;         // num_draft[b]
    bool greedy;
    float kappa;   // log2(e) / T
    int xj;        // draft token of the row (-1: none, or out of range)
    int xchunk;    // chunk holding xj (-1: none)
};

__device__ __forceinline__ RowCtx row_ctx(const Params& P, int slot) {
    RowCtx rc;
    rc.slot = slot;
    const int b = rc.slot / P.K1, j = rc.slot - b * P.K1;
    rc.b = b;
    rc.n = P.num_draft[b];
    const float T = P.temp[b];
    rc.greedy = (T == 0.f);
    rc.kappa = rc.greedy ? 0.f : kappa_of(T);
    int x = -1;
    if (!P.tree && !rc.greedy && j < rc.n) {  // tree requests gather nothing here
        x = P.ids[(size_t)b * P.K + j];
        if (x < 0 || x >= P.V) x = -1;  // reported by the acceptance step
    }
    rc.xj = x;
    rc.xchunk = x >= 0 ? x / TILE : -1;
    return rc;
}
__device__ __forceinline__ RowCtx row_ctx(const Params& P, const int* rowlist, long long r) {
    return row_ctx(P, rowlist[r]);
}

}  // namespace



// The all-rows pass (and a tree pass), balanced across SMs.  The streaming
// speed of a warp depends on where its SM sits (measured: warps of an equal
// static split ended between 29 and 44 us on the largest-vocabulary workload,
// the same SMs slow in every run), so an equal split leaves a tail.  Warp w
// streams the first 7/8 of its equal range [T w / W, T (w + 1) / W) as a
// static segment, and the last 1/8 of every range is handed out as one
// segment per claim: claim k (one atomic on a counter k_plan cleared, fired
// a few tiles before the claimer runs out of work, so in about the order in
// which warps finish) takes the tail of warp (k * CLAIM_STRIDE) mod W; the
// stride is a prime above any warp count, so the claims take every tail
// exactly once and consecutive claims land far apart in the logits.  The
// producer lane passes each staged tile's row slot and chunk to the
// consumer through shared memory, with the tiles left in its segment.
#ifndef SV_TAIL_DEN
#define SV_TAIL_DEN 8
#endif
#ifndef SV_FIRE_AHEAD
#define SV_FIRE_AHEAD 2
#endif
constexpr int TAIL_DEN = SV_TAIL_DEN;        // the claimed tail is 1/TAIL_DEN of each range
constexpr long long CLAIM_STRIDE = 1000003;  // prime
constexpr int FIRE_AHEAD = SV_FIRE_AHEAD;    // tiles left when the next claim goes out

template <int DT>
__device__ __forceinline__ void stream_balanced(const Params& P, uint8_t* buf,
                                                uint64_t (*bars)[STATS_STAGES], const int* rowlist,
                                                long long T, long long W, long long w) {
    using TL = Tile<DT>;
    constexpr int EPV = TL::EPV, VPL = TL::VPL;
    __shared__ int4 sinfo[STATS_WARPS][STATS_STAGES];  // {slot, chunk, tiles left in segment, segment start}
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = P.C;

    // ---- producer state (lane 0)
    const long long t0 = T * w / W, t1 = T * (w + 1) / W;
    long long pt = t0, pe = t1 - (t1 - t0) / TAIL_DEN;  // the static segment
    bool seg_first = true;  // the next issued tile starts a segment
    bool fired = false;     // a claim is in flight for the next segment
    int claim = 0;
    bool done = false;
    int issued = 0;
    long long prow = -1;
    int pslot = 0;
    auto fire = [&]() {
        claim = atomicAdd(P.hdr + HDR_CLAIM, 1);
        fired = true;
    };
    // lane 0: move to the next claimed tail; false when every tail is taken
    auto next_segment = [&]() -> bool {
        for (;;) {
            if (!fired) fire();
            fired = false;
            if (claim >= W) return false;
            const long long v = ((long long)claim * CLAIM_STRIDE) % W;
            const long long a = T * v / W, b = T * (v + 1) / W;
            const long long tail = (b - a) / TAIL_DEN;
            if (tail > 0) {
                pt = b - tail;
                pe = b;
                seg_first = true;
                return true;
            }
        }
    };
    auto issue = [&](int s) {
        if (done) return;
        while (pt == pe)
            if (!next_segment()) {
                done = true;
                return;
            }
        if (!fired && pe - pt <= FIRE_AHEAD) fire();
        const long long r = pt / C;
        const int c = int(pt - r * C);
        if (r != prow) {
            prow = r;
            pslot = rowlist[r];
        }
        const int nel = min(TILE, P.V - c * TILE);
        const uint32_t bytes = uint32_t(nel) * TL::ESZ;
        const char* src = reinterpret_cast<const char*>(P.logits) +
                          ((size_t)pslot * P.V + (size_t)c * TILE) * TL::ESZ;
        sinfo[warp][s] = make_int4(pslot, c, int(pe - pt - 1), seg_first ? 1 : 0);
        seg_first = false;
        mbar_arrive_expect_tx(&bars[warp][s], bytes);
        bulk_g2s(buf + s * TL::BYTES, src, bytes, &bars[warp][s]);
        ++pt;
        ++issued;
    };
    if (lane == 0)
        for (int k = 0; k < STATS_STAGES; ++k) issue(k);

    // ---- consumer (whole warp)
    RowCtx rc;
    rc.slot = -1;
    float qx = 0.f;
    long long i = 0;
    int s = 0;
    uint32_t parity = 0;
    bool timed_out = false;
    int have = 0;
    for (;; ++i) {
        have = __shfl_sync(0xffffffffu, issued, 0);
        if (i >= have) break;
        const bool landed = mbar_wait_bounded(&bars[warp][s], parity);
        if (!__all_sync(0xffffffffu, landed)) {  // warp-uniform exit
            timed_out = true;
            break;
        }
        const int4 si = sinfo[warp][s];
        const int cc = si.y;
        if (si.x != rc.slot || si.w) {
            if (si.x != rc.slot) rc = row_ctx(P, si.x);
            // q_j(x_j) is fetched by the warp whose segment holds x_j's tile
            if (P.rule == RULE_LOSSLESS && rc.xj >= 0 && rc.xchunk >= cc &&
                rc.xchunk - cc <= si.z && lane == 0) {
                const int b = rc.slot / P.K1, j = rc.slot - b * P.K1;
                qx = __ldg(P.probs + ((size_t)b * P.K + j) * P.V + rc.xj);
            }
        }
        const int nvec = min(TILE, P.V - cc * TILE) / EPV;
        const uint8_t* stage = buf + s * TL::BYTES;
        const uint4* v4 = reinterpret_cast<const uint4*>(stage);
        uint4 d[VPL];
        if (nvec == TILE / EPV) {
#pragma unroll
            for (int k = 0; k < VPL; ++k) d[k] = v4[k * 32 + lane];
        } else {  // the row's ragged last chunk: pad with -inf
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int v = k * 32 + lane;
                d[k] = v < nvec ? v4[v]
                                : make_uint4(TL::NEG_INF_WORD, TL::NEG_INF_WORD,
                                             TL::NEG_INF_WORD, TL::NEG_INF_WORD);
            }
        }
        const bool has_x = (cc == rc.xchunk);
        float lx = 0.f;
        if (has_x && lane == 0) {
            const int e = rc.xj - cc * TILE;
            if constexpr (DT == SPEC_BF16)
                lx = __uint_as_float(uint32_t(reinterpret_cast<const uint16_t*>(stage)[e]) << 16);
            else
                lx = reinterpret_cast<const float*>(stage)[e];
        }
        __syncwarp();  // every lane holds its share: the stage can be refilled
        if (lane == 0) {
            fence_proxy_async_smem();
            issue(s);
        }
        const Partial out = tile_partial<DT>(d, nvec, cc * TILE, rc.greedy, rc.kappa);
        if (lane == 0) {
            P.part[(size_t)rc.slot * C + cc] = out;
            if (has_x) P.gath[rc.slot] = make_float2(lx, qx);
        }
        if (++s == STATS_STAGES) {
            s = 0;
            parity ^= 1u;
        }
    }
    if (timed_out) {
        if (lane == 0) atomicOr(P.status, int(SPEC_BADBIT_TIMEOUT));
        // let the copies still in flight land before the CTA's shared memory is released
        for (long long u = i; u < have && u < i + STATS_STAGES; ++u)
            mbar_wait_bounded(&bars[warp][int(u % STATS_STAGES)], uint32_t((u / STATS_STAGES) & 1),
                              100000000ull);
    }
}

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

    // the rows of this pass: all of them, or those of one early-exit round
    const bool later_round = P.round > 0;
    const int* rowlist = later_round ? P.rowlist + (size_t)P.round * P.B : P.rowlist;
    const long long R = later_round ? __ldcg(P.hdr + HDR_ROUND + P.round) : P.hdr[HDR_ROWS];
    const long long T = R * P.C;
    const long long W = (long long)gridDim.x * STATS_WARPS;
    const long long w = (long long)blockIdx.x * STATS_WARPS + warp;
    if (P.round < 0) {  // the all-rows pass: balanced across SMs
        stream_balanced<DT>(P, buf, bars, rowlist, T, W, w);
        return;
    }
    const long long t0 = T * w / W, t1 = T * (w + 1) / W;
    if (t0 >= t1) return;
    const long long r0 = t0 / P.C;
    const int c0 = int(t0 - r0 * P.C);
    const long long n_tiles = t1 - t0;

    // producer (lane 0): next tile to issue, as (row, chunk), and its row's slot
    long long pr = r0;
    int pc = c0;
    int pslot = lane == 0 ? rowlist[r0] : 0;
    auto issue = [&](int s) {
        const int nel = min(TILE, P.V - pc * TILE);
        const uint32_t bytes = uint32_t(nel) * TL::ESZ;
        const char* src = reinterpret_cast<const char*>(P.logits) +
                          ((size_t)pslot * P.V + (size_t)pc * TILE) * TL::ESZ;
        mbar_arrive_expect_tx(&bars[warp][s], bytes);
        bulk_g2s(buf + s * TL::BYTES, src, bytes, &bars[warp][s]);
        if (++pc == P.C) {
            pc = 0;
            if (++pr < R) pslot = rowlist[pr];
        }
    };
    if (lane == 0) {
        for (int k = 0; k < STATS_STAGES && k < n_tiles; ++k) issue(k);
    }

    // consumer state
    long long cr = r0;
    int cc = c0;
    RowCtx rc = row_ctx(P, rowlist, cr);
    float qx = 0.f;  // q_j(x_j), fetched at row start by the warp that owns x_j's tile
    auto prefetch_q = [&]() {
        const long long t_x = cr * P.C + rc.xchunk;
        if (P.rule == RULE_LOSSLESS && rc.xj >= 0 && t_x >= t0 && t_x < t1 && lane == 0) {
            const int b = rc.slot / P.K1, j = rc.slot - b * P.K1;
            qx = __ldg(P.probs + ((size_t)b * P.K + j) * P.V + rc.xj);
        }
    };
    prefetch_q();

    // the run of consecutive tiles of one request that this warp has finished
    int seg_b = rc.b, seg_n = rc.n, seg_tiles = 0;
    bool seg_greedy = rc.greedy;
    float seg_kappa = rc.kappa;
    // Only early-exit passes count tiles here: the all-rows pass leaves every
    // acceptance to k_accept_all, so its warps never stop streaming to fence
    // and count (a warp whose range crossed a request boundary used to lose
    // about 5 us there), and tree passes are walked by k_tree_walk.
    const bool counting = P.round >= 0 && !P.tree;
    auto flush = [&]() {
        int last = 0;
        if (lane == 0 && seg_tiles > 0 && counting) {
            __threadfence();  // this warp's partials before its count
            // an early-exit request completes one row per round; its count
            // is never reset, so round r ends at (r + 1) * C
            const int total = (P.round >= 0 ? P.round + 1 : seg_n + 1) * P.C;
            last = atomicAdd(&P.cnt[seg_b], seg_tiles) + seg_tiles == total;
        }
        if (__shfl_sync(0xffffffffu, last, 0)) {
            __threadfence();  // every other warp's partials after the count
            accept_request(P, seg_b, seg_n, seg_greedy, seg_kappa);
        }
        seg_tiles = 0;
    };

    long long i = 0;
    int s = 0;            // stage of tile i
    uint32_t parity = 0;  // phase of that stage's barrier
    bool timed_out = false;
    for (; i < n_tiles; ++i) {
        const int nvec = min(TILE, P.V - cc * TILE) / EPV;

        const bool landed = mbar_wait_bounded(&bars[warp][s], parity);
        if (!__all_sync(0xffffffffu, landed)) {  // warp-uniform exit
            timed_out = true;
            break;
        }
        const uint8_t* stage = buf + s * TL::BYTES;
        const uint4* v4 = reinterpret_cast<const uint4*>(stage);
        uint4 d[VPL];
        if (nvec == TILE / EPV) {  // full tile
#pragma unroll
            for (int k = 0; k < VPL; ++k) d[k] = v4[k * 32 + lane];
        } else {                   // the row's ragged last chunk: pad with -inf
#pragma unroll
            for (int k = 0; k < VPL; ++k) {
                const int v = k * 32 + lane;
                d[k] = v < nvec ? v4[v]
                                : make_uint4(TL::NEG_INF_WORD, TL::NEG_INF_WORD,
                                             TL::NEG_INF_WORD, TL::NEG_INF_WORD);
            }
        }
        const bool has_x = (cc == rc.xchunk);
        float lx = 0.f;
        if (has_x && lane == 0) {
            const int e = rc.xj - cc * TILE;
            if constexpr (DT == SPEC_BF16)
                lx = __uint_as_float(uint32_t(reinterpret_cast<const uint16_t*>(stage)[e]) << 16);
            else
                lx = reinterpret_cast<const float*>(stage)[e];
        }
        __syncwarp();  // every lane holds its share: the stage can be refilled
        if (lane == 0 && i + STATS_STAGES < n_tiles) {  // tile i + STAGES reuses stage s
            fence_proxy_async_smem();
            issue(s);
        }

        const Partial out = tile_partial<DT>(d, nvec, cc * TILE, rc.greedy, rc.kappa);
        if (lane == 0) {
            P.part[(size_t)rc.slot * P.C + cc] = out;
            if (has_x) P.gath[rc.slot] = make_float2(lx, qx);
        }
        ++seg_tiles;
        if (++cc == P.C) {
            cc = 0;
            if (++cr < R && i + 1 < n_tiles) {
                rc = row_ctx(P, rowlist, cr);
                prefetch_q();
                if (rc.b != seg_b) {  // the warp moves on to the next request
                    flush();
                    seg_b = rc.b;
                    seg_n = rc.n;
                    seg_greedy = rc.greedy;
                    seg_kappa = rc.kappa;
                }
            }
        }
        if (++s == STATS_STAGES) {
            s = 0;
            parity ^= 1u;
        }
    }

    if (!timed_out) flush();
    if (timed_out) {
        if (lane == 0) atomicOr(P.status, int(SPEC_BADBIT_TIMEOUT));
        // let the copies still in flight land before the CTA's shared memory is released
        for (long long u = i; u < n_tiles && u < i + STATS_STAGES; ++u)
            mbar_wait_bounded(&bars[warp][int(u % STATS_STAGES)], uint32_t((u / STATS_STAGES) & 1),
                              100000000ull);
    }
}

// The acceptance of every valid request once all its row statistics exist
// (after the all-rows pass, or after the fused projection): one CTA per
// request; its warps merge the request's rows side by side (warp w: rows w,
// w + ACCEPT_WARPS, ...), then warp 0, whose own loads were issued first,
// decides.
__global__ void __launch_bounds__(ACCEPT_WARPS * 32) k_accept_all(Params P) {
    griddep_launch_dependents();
    griddep_wait();  // the row statistics
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (b >= P.B) return;
    __shared__ float s_m[SPEC_MAX_K + 1], s_z[SPEC_MAX_K + 1];
    __shared__ int s_a[SPEC_MAX_K + 1];
    // Loads that need nothing loaded first go out together with num_draft
    // and temperature: each warp's first row of partials, and warp 0's draft
    // tokens, gathers and Philox blocks for every row the request may have
    // (rows past num_draft are never used).
    const Partial* pb = P.part + (size_t)b * P.K1 * P.C;
    Partial q0[MERGE_NPL];
    const bool pre = P.C <= 32 * MERGE_NPL && warp < P.K1;
    if (pre) load_row(pb + (size_t)warp * P.C, P.C, q0);
    AccLoads L;
    if (warp == 0) L = accept_loads(P, b, P.K, false, 0, P.K);
    const int flags = P.req_flags[b];
    const int n = P.num_draft[b];
    const float T = P.temp[b];
    if (flags != 0) return;  // bad requests: k_plan wrote their outputs
    const bool greedy = (T == 0.f);
    const float kappa = greedy ? 0.f : kappa_of(T);
    for (int j = warp; j <= n; j += ACCEPT_WARPS) {
        float M, Z;
        int A;
        if (j == warp && pre)
            merge_loaded(q0, greedy, kappa, M, Z, A);
        else
            merge_row(pb + (size_t)j * P.C, P.C, greedy, kappa, M, Z, A);
        if (lane == 0) {
            s_m[j] = M;
            s_z[j] = Z;
            s_a[j] = A;
        }
    }
    __syncthreads();
    if (warp == 0) {
        const bool mine = lane <= n;
        accept_decide(P, b, n, greedy, kappa, L, mine ? s_m[lane] : -INFINITY,
                      mine ? s_a[lane] : INT_MAX, mine ? s_z[lane] : 0.f);
    }
}

__global__ void __launch_bounds__(STATS_WARPS * 32) k_row_stats_f32(Params P) {
    row_stats_body<SPEC_F32>(P);
}
__global__ void __launch_bounds__(STATS_WARPS * 32) k_row_stats_bf16(Params P) {
    row_stats_body<SPEC_BF16>(P);
}

}  // namespace sv
