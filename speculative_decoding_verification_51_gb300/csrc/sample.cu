// sample.cu -- k_sample: the emitted token of every sampling request.
//
// Residual ("深入推测解码" 保证原始分布 step 4; "投机采样" 第四步 and 第五步):
// at the first rejected row e the token is drawn from norm(max(0, p_e - q_e)).
// Bonus ("投机采样" output-length case 3): when all drafts are accepted one token
// is drawn from p_{n_b}.  Both draws are an inverse CDF with the row's emission
// uniform u' (Philox lane 1): the smallest x with C(x) >= u' * C(V-1), C the
// prefix sum of the weights in token order.
//
// The CDF is evaluated in two levels so that only one 2048-token chunk is ever
// scanned:
//   level 1: per-chunk masses (residual: summed here, one warp per chunk;
//            bonus: the row-stat partials of k_row_stats), prefix-summed in
//            float64 in chunk order -> the chunk c* holding u' * C(V-1);
//   level 2: the chunk c* is copied into shared memory, its weights recomputed
//            with the same float32 expression as level 1, and scanned in token
//            order (8-token groups, float32): the first token whose running sum
//            reaches the remaining mass is taken.  Tokens of zero mass are
//            never taken; if rounding leaves the threshold beyond the chunk,
//            its last token of positive mass is.
// Every unit of work belongs to one warp and warps never wait for each other.
// k_sample: a residual unit is one chunk of (logits row, draft row) whose mass
// is stored; a pair of warps copies the chunk into shared memory with two 1-D
// bulk copies (cp.async.bulk, mbarrier completion) while the previous unit is
// being reduced (two stages per pair), each warp reducing half its groups.  k_emit (the next kernel, once the memory
// system is free of the streaming traffic): one warp per draw, residual or
// bonus, runs both levels.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "draw.cuh"

namespace sv {

namespace {

// The per-warp double-buffered staging area.
struct WarpStages {
    uint8_t* base;      // stage s starts at base + s * stage_bytes
    uint64_t* bars;     // bars[s]
    int stage_bytes;
    uint32_t phase;     // bit s: phase of stage s's barrier
    uint32_t inflight;  // bit s: a copy into stage s has not been waited for
    bool broken;        // a bounded wait gave up

    __device__ __forceinline__ uint8_t* buf(int s) const { return base + s * stage_bytes; }

    // lane 0: copy `bl` bytes of logits (and `bq` of q) into stage s
    __device__ __forceinline__ void issue(int s, const void* l, uint32_t bl, const void* q,
                                          uint32_t bq, int lb_offset) {
        if ((threadIdx.x & 31) == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(bars + s, bl + bq);
            bulk_g2s(buf(s), l, bl, bars + s);
            if (bq) bulk_g2s(buf(s) + lb_offset, q, bq, bars + s);
        }
        inflight |= 1u << s;
    }
    // whole warp: wait for stage s (bounded); false if the wait gave up, and
    // then the copy still counts as in flight
    __device__ __forceinline__ bool wait(int s) {
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bars + s, (phase >> s) & 1u));
        if (ok) {
            phase ^= 1u << s;
            inflight &= ~(1u << s);
        }
        return ok;
    }
};

__device__ __forceinline__ void write_emit(const Params& P, const ReqRec& rec, int x, int mode,
                                           double mass) {
    if ((threadIdx.x & 31) != 0) return;
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
// residual when it has no mass).  Level 2 stages the chunk in stage s.
template <int DT>
__device__ __forceinline__ void emit_from_p(const Params& P, const ReqRec& rec, int mode,
                                            WarpStages& ws, int s) {
    const Partial* part = P.part + ((size_t)rec.b * P.K1 + rec.erow) * P.C;
    const float m = rec.m, kappa = rec.kappa;
    const Pick pk = pick_chunk(P.C, rec.u2, [&](int c) -> double {
        const Partial q = part[c];
        if (q.m == -INFINITY || q.z == 0.0) return 0.0;
        return q.z * double(rebase_factor(q.m, m, kappa));
    });
    if (pk.chunk < 0) {  // no mass at all (cannot happen for a row with a finite logit)
        write_emit(P, rec, 0, mode, pk.total);
        return;
    }
    const Partial pc = part[pk.chunk];
    const double f_c = double(rebase_factor(pc.m, m, kappa));
    const double t = (double(rec.u2) * pk.total - pk.before) * pow2_recip(f_c);  // chunk-local
    const float cc = offset_of(pc.m, kappa);
    const int c0 = pk.chunk * TILE, nel = min(TILE, P.V - c0);
    const char* src = reinterpret_cast<const char*>(P.logits) +
                      (((size_t)rec.b * P.K1 + rec.erow) * P.V + c0) * Stage<DT>::ESZ;
    ws.issue(s, src, uint32_t(nel) * Stage<DT>::ESZ, nullptr, 0, Stage<DT>::LB);
    if (!ws.wait(s)) {
        ws.broken = true;
        return;
    }
    const uint8_t* st = ws.buf(s);
    const int x = level2(c0, nel, t, [&](int g, float (&w)[8]) {
        float l[8];
        smem_logits8<DT>(st, g, l);
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = ex2_approx(weight_arg(l[k], pc.m, cc, kappa));
    });
    __syncwarp();
    write_emit(P, rec, x, mode, pk.total);
}

// One warp's share of the residual mass of a staged chunk of nel tokens.  The
// chunk's 8-token groups are k * 32 + l (lane l, k = 0..7, coalesced); warp
// `odd` of the pair takes k = odd, odd + 2, odd + 4, odd + 6, sums each
// group's 8 weights pairwise in float32, then (k, k + 4) pairs and the two
// pair sums.  The even warp's value plus the odd warp's, summed over the lanes,
// is the pairwise sum of the lane's 8 groups.  FIN: the row offset passes
// offset_ok (the weight exponent is then one FFMA, as weight_arg computes it).
template <int DT, bool FIN>
__device__ __forceinline__ float staged_residual_half(const uint8_t* st, int nel,
                                                      const ReqRec& rec, int odd) {
    const int lane = threadIdx.x & 31;
    const float invZ = float(1.0 / rec.Z);
    const float cm = offset_of(rec.m, rec.kappa);
    float gs[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int g = (2 * t + odd) * 32 + lane;
        gs[t] = 0.f;
        if (g * 8 < nel) {
            float l[8], q[8];
            smem_logits8<DT>(st, g, l);
            smem_q8(st + Stage<DT>::LB, g, q);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float arg = FIN ? fmaf(l[e], rec.kappa, -cm)
                                      : __fmul_rn(__fsub_rn(l[e], rec.m), rec.kappa);
                const float p = __fmul_rn(ex2_approx(arg), invZ);
                l[e] = fmaxf(__fsub_rn(p, q[e]), 0.f);
            }
#pragma unroll
            for (int h = 4; h; h >>= 1)
#pragma unroll
                for (int e = 0; e < h; ++e) l[e] = __fadd_rn(l[e], l[e + h]);
            gs[t] = l[0];
        }
    }
    return __fadd_rn(__fadd_rn(gs[0], gs[2]), __fadd_rn(gs[1], gs[3]));
}

// bar.red.and over the 64 threads of warp pair `pair` (named barrier 1 + pair):
// true iff every thread's `ok` is; also orders the pair's shared-memory accesses.
// The barrier number is a literal in each case so that only the barriers in use
// are reserved.
template <int ID>
__device__ __forceinline__ bool bar_red_and64(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "barrier.red.and.pred po, %2, 64, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(uint32_t(ok)), "n"(ID)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool pair_and(int pair, bool ok) {
    static_assert(SAMPLE_PAIRS <= 8, "one named barrier per pair");
    switch (pair) {
        case 0: return bar_red_and64<1>(ok);
        case 1: return bar_red_and64<2>(ok);
        case 2: return bar_red_and64<3>(ok);
        case 3: return bar_red_and64<4>(ok);
        case 4: return bar_red_and64<5>(ok);
        case 5: return bar_red_and64<6>(ok);
        case 6: return bar_red_and64<7>(ok);
        default: return bar_red_and64<8>(ok);
    }
}

// Level 1 and 2 of the residual of queued request i.  pre: the chunk masses
// as load_masses holds them, loaded by the caller when C <= PICK_NB * 32.
// Level 2 stages the chunk in stage s.
template <int DT>
__device__ __forceinline__ void emit_residual(const Params& P, const ReqRec& rec, int i,
                                              const double (&pre)[PICK_NB], WarpStages& ws,
                                              int s) {
    const float* rs = P.rsum + (size_t)i * P.C;
    const Pick pk = P.C <= PICK_NB * 32
                        ? pick_loaded(rec.u2, pre)
                        : pick_chunk(P.C, rec.u2, [&](int c) -> double { return double(__ldcg(rs + c)); });
    if (pk.chunk < 0) {  // residual without mass: draw from p instead
        emit_from_p<DT>(P, rec, MODE_FALLBACK, ws, s);
        return;
    }
    const double t = double(rec.u2) * pk.total - pk.before;
    const float invZ = float(1.0 / rec.Z);
    const float cm = offset_of(rec.m, rec.kappa);
    const int c0 = pk.chunk * TILE, nel = min(TILE, P.V - c0);
    const char* l = reinterpret_cast<const char*>(P.logits) +
                    (((size_t)rec.b * P.K1 + rec.erow) * P.V + c0) * Stage<DT>::ESZ;
    const float* q = P.probs + ((size_t)rec.b * P.K + rec.erow) * P.V + c0;
    ws.issue(s, l, uint32_t(nel) * Stage<DT>::ESZ, q, uint32_t(nel) * 4u, Stage<DT>::LB);
    if (!ws.wait(s)) {
        ws.broken = true;
        return;
    }
    const uint8_t* st = ws.buf(s);
    const int x = level2(c0, nel, t, [&](int g, float (&w)[8]) {
        float lv[8], qv[8];
        smem_logits8<DT>(st, g, lv);
        smem_q8(st + Stage<DT>::LB, g, qv);
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = resid(lv[k], qv[k], rec.m, cm, rec.kappa, invZ);
    });
    __syncwarp();
    write_emit(P, rec, x, MODE_RESIDUAL, pk.total);
}

}  // namespace

// Per-warp staging setup.
template <int DT>
__device__ __forceinline__ WarpStages make_stages(uint8_t* smem, uint64_t* bars, int nstages) {
    using ST = Stage<DT>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WarpStages ws;
    ws.base = smem + size_t(warp) * nstages * ST::BYTES;
    ws.bars = bars + warp * 2;
    ws.stage_bytes = ST::BYTES;
    ws.phase = 0;
    ws.inflight = 0;
    ws.broken = false;
    if (lane == 0) {
        for (int k = 0; k < nstages; ++k) mbar_init(ws.bars + k, 1);
        fence_mbarrier_init();
    }
    __syncwarp();
    return ws;
}

__device__ __forceinline__ void finish_stages(const Params& P, WarpStages& ws) {
    if (ws.broken) {
        if ((threadIdx.x & 31) == 0) atomicOr(P.status, int(SPEC_BADBIT_TIMEOUT));
        // let copies still in flight land before the CTA's shared memory is released
        for (int k = 0; k < 2; ++k)
            if (ws.inflight & (1u << k))
                mbar_wait_bounded(ws.bars + k, (ws.phase >> k) & 1u, 100000000ull);
    }
}

// k_sample: the residual chunk masses of every queued request.  Each pair of
// warps takes an equal contiguous range of the units (queue entry i, chunk c)
// in order and keeps SAMPLE_STAGES staging buffers: the bulk copies of the
// next SAMPLE_STAGES - 1 chunks (issued by the even warp) are in flight while
// both warps reduce the current one.  Sharing each chunk between two warps
// doubles the warps per SM for the same shared memory.  A pure streaming
// pass: the draws themselves are made by k_emit.
template <int DT>
__device__ __forceinline__ void sample_body(const Params& P) {
    using ST = Stage<DT>;
    constexpr int NS = SAMPLE_STAGES;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[SAMPLE_PAIRS * NS];
    __shared__ float xch[SAMPLE_PAIRS][NS][32];  // the odd warp's lane sums, per stage
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pair = warp >> 1, odd = warp & 1;
    WarpStages ws;
    ws.base = smem + size_t(pair) * NS * ST::BYTES;
    ws.bars = bars + pair * NS;
    ws.stage_bytes = ST::BYTES;
    ws.phase = 0;
    ws.inflight = 0;
    ws.broken = false;
    if (threadIdx.x < SAMPLE_PAIRS * NS) {
        mbar_init(bars + threadIdx.x, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    griddep_launch_dependents();
    griddep_wait();  // decisions and queues of the acceptance step
    const int C = P.C;
    const long long W = (long long)gridDim.x * SAMPLE_PAIRS;
    const long long pid = (long long)blockIdx.x * SAMPLE_PAIRS + pair;
    const long long VT = (long long)P.hdr[HDR_NRES] * C;
    const long long r0 = VT * pid / W, r1 = VT * (pid + 1) / W;
    if (r0 < r1) {  // uniform over the pair
        ReqRec cur = P.res_rec[r0 / C];
        // producer (even warp): the next unit to copy, its record and stage
        long long pv = r0;
        ReqRec prec = cur;
        int ps = 0;
        auto issue_next = [&]() {
            if (odd || pv >= r1) return;
            const int c = int(pv % C);
            const int c0 = c * TILE, nel = min(TILE, P.V - c0);
            const char* l = reinterpret_cast<const char*>(P.logits) +
                            (((size_t)prec.b * P.K1 + prec.erow) * P.V + c0) * ST::ESZ;
            const float* q = P.probs + ((size_t)prec.b * P.K + prec.erow) * P.V + c0;
            ws.issue(ps, l, uint32_t(nel) * ST::ESZ, q, uint32_t(nel) * 4u, ST::LB);
            ps = ps + 1 == NS ? 0 : ps + 1;
            if (++pv < r1 && pv % C == 0) prec = P.res_rec[pv / C];
        };
#pragma unroll
        for (int k = 0; k < NS - 1; ++k) issue_next();
        int s = 0;
        for (long long v = r0; v < r1; ++v) {
            // the stage read at the last pair barrier is refilled first
            issue_next();
            const bool ok = ws.wait(s);
            // a stage that did not land is still read (in bounds) but its sum is dropped
            const int c = int(v % C);
            const int nel = min(TILE, P.V - c * TILE);
            const float part = offset_ok(offset_of(cur.m, cur.kappa))
                                   ? staged_residual_half<DT, true>(ws.buf(s), nel, cur, odd)
                                   : staged_residual_half<DT, false>(ws.buf(s), nel, cur, odd);
            if (odd) xch[pair][s][lane] = part;
            if (!pair_and(pair, ok)) {  // the same decision in both warps
                ws.broken = true;
                break;
            }
            if (!odd) {
                const float sum = warp_sum_f(__fadd_rn(part, xch[pair][s][lane]));
                if (lane == 0) P.rsum[v] = sum;  // entry v / C, chunk c
            }
            if (v + 1 < r1 && (v + 1) % C == 0) cur = P.res_rec[(v + 1) / C];
            s = s + 1 == NS ? 0 : s + 1;
        }
    }
    finish_stages(P, ws);  // the even warp waits for its copies still in flight
}

// k_emit: one warp per queue slot once every residual mass exists: even
// warps take the residual queue's slots, odd warps the bonus queue's (draws
// from p), so that the filled slots of both queues spread over the SMs (the
// draws' float64 steps share an SM's narrow FP64 pipe).  A warp loads its
// slot's count, record and (residual) chunk masses together, all in bounds
// whether or not the slot is filled, and leaves if it is not: no load of the
// draw waits for another.
template <int DT>
__device__ __forceinline__ void emit_body(const Params& P) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[EMIT_WARPS * 2];
    WarpStages ws = make_stages<DT>(smem, bars, 1);
    griddep_launch_dependents();
    griddep_wait();  // chunk masses of k_sample
    const long long w = (long long)blockIdx.x * EMIT_WARPS + (threadIdx.x >> 5);
    const bool res = (w & 1) == 0;
    const int slot = int(w >> 1);
    if (slot >= P.B) return;  // grid rounding (warp-uniform)
    const int count = P.hdr[res ? HDR_NRES : HDR_NBONUS];
    // the record is copied to registers: every step of the draw reads it
    const ReqRec r = res ? P.res_rec[slot] : P.bonus_rec[slot];
    double pre[PICK_NB];
    if (res && P.C <= PICK_NB * 32) {
        const float* rs = P.rsum + (size_t)slot * P.C;
        load_masses(P.C, [&](int c) -> double { return double(__ldcg(rs + c)); }, pre);
    }
    if (slot >= count) return;
    if (res)
        emit_residual<DT>(P, r, slot, pre, ws, 0);
    else
        emit_from_p<DT>(P, r, r.mode, ws, 0);
    finish_stages(P, ws);
}

__global__ void __launch_bounds__(SAMPLE_PAIRS * 64) k_sample_f32(Params P) {
    sample_body<SPEC_F32>(P);
}
__global__ void __launch_bounds__(SAMPLE_PAIRS * 64) k_sample_bf16(Params P) {
    sample_body<SPEC_BF16>(P);
}
__global__ void __launch_bounds__(EMIT_WARPS * 32) k_emit_f32(Params P) { emit_body<SPEC_F32>(P); }
__global__ void __launch_bounds__(EMIT_WARPS * 32) k_emit_bf16(Params P) { emit_body<SPEC_BF16>(P); }


}  // namespace sv
