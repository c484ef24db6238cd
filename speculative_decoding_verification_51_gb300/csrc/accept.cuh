// accept.cuh -- acceptance of one request by one warp: in k_accept_all (one
// warp per request) once the all-rows pass or the fused projection has
// written every row statistic, and inside k_row_stats, by the warp that
// completes a request's row, in an early-exit pass.
//
// Lane j owns row j of the request.  Steps (pages cited by title / section):
//   1. merge the chunk partials of every row j <= n_b into the row's max m_j,
//      normaliser Z_j = sum_x 2^((l_j(x) - m_j) kappa) and, for greedy rows,
//      the lowest-index argmax (merge_row: one warp per row, float32
//      throughout: the FP64 pipe of this part is slow);
//   2. acceptance of draft x_j ("深入推测解码" 保证原始分布 step 3,
//      "RTP-LLM Speculative Engine" 拒绝采样算法): p = 2^((l_j(x_j) - m_j) kappa)
//      / Z_j with l_j(x_j) and q_j(x_j) gathered by k_row_stats, u_j = Philox
//      lane 0 of row j; accept iff p > 0 and (q_j(x_j) == 0 or
//      u_j <= p / q_j(x_j)), tested exactly as u q <= p in float64; greedy
//      ("投机采样" 精确匹配): accept iff x_j is the row's argmax;
//   3. first-reject scan in-warp: a_b = position of the lowest zero of the
//      ballot of acceptance bits ("投机采样" 第五步: drafts after a rejected
//      one are discarded);
//   4. write the accepted prefix and the -1 tail; greedy requests also write
//      the emitted token (argmax of row a_b); sampling requests are queued for
//      k_sample (residual at row a_b < n_b, bonus at row a_b == n_b).
// Under the typical-acceptance rule ("投机采样" 验收标准, Typical Acceptance)
// step 2 keeps x_j iff p > 0 and p >= the call's threshold (no q, no u_j) and
// every sampling request is queued as a draw from p at row a_b.
// Early exit (P.round = r >= 0): the pass holds row r only, and every earlier
// draft of the request was kept.  The same steps run on that one row: a kept
// draft is written out and row r + 1 joins the list of the next round;
// otherwise the request ends here with a_b = r, exactly as the all-rows pass
// would have ended it.
// Partials and gathers written by other warps are read through L2
// (ld.global.cg): after the caller's fence (early exit) or in the next kernel.
#pragma once

#include <cfloat>
#include <climits>

#include "common.cuh"

namespace sv {

namespace {

// (m, z) <- (m, z) (+) (m2, z2): sums of 2^((l - m) kappa) with different maxima.
__device__ __forceinline__ void merge_sum(float& m, float& z, float m2, float z2, float kappa) {
    if (m2 > m) {
        const float tm = m;
        m = m2;
        m2 = tm;
        const float tz = z;
        z = z2;
        z2 = tz;
    }
    if (m2 != -INFINITY && z2 != 0.f) z = fmaf(z2, rebase_factor(m2, m, kappa), z);
}

__device__ __forceinline__ void merge_argmax(float& m, int& a, float m2, int a2) {
    if (m2 > m || (m2 == m && a2 < a)) {
        m = m2;
        a = a2;
    }
}

}  // namespace

// The per-lane inputs of the acceptance that depend on nothing merged: the
// draft token, its gathered {l_j(x_j), q_j(x_j)} and the Philox block of the
// lane's row (rows jlo..jhi of request b).
struct AccLoads {
    int x;
    float2 g;
    uint4 rb;
};

__device__ __forceinline__ AccLoads accept_loads(const Params& P, int b, int n, bool greedy,
                                                 int jlo, int jhi) {
    const int lane = threadIdx.x & 31;
    const bool row_lane = lane >= jlo && lane <= jhi;
    const bool draft_lane = row_lane && lane < n;
    AccLoads L;
    L.x = draft_lane ? P.ids[(size_t)b * P.K + lane] : -1;
    L.g = make_float2(0.f, 0.f);
    if (draft_lane && !greedy) L.g = __ldcg(P.gath + (size_t)b * P.K1 + lane);
    L.rb = make_uint4(0, 0, 0, 0);
    if (!greedy && row_lane) L.rb = row_block(P, b, lane);
    return L;
}

// Step 1 for one row (whole warp; every lane gets the result): M = the row
// max, Z = its normaliser against offset_of(M, kappa), A = the lowest index of the
// max (greedy rows).  With at most 128 chunks a lane's chunks stay in
// registers: the max first (shuffles), then every chunk rebased onto it once
// (one ex2 each) and summed (shuffles); longer rows merge pairwise.
constexpr int MERGE_NPL = 4;  // chunks per lane held in registers (rows of up to 128 chunks)

// This lane's chunk partials of a row of C <= 32 * MERGE_NPL chunks.
__device__ __forceinline__ void load_row(const Partial* prow, int C, Partial (&q)[MERGE_NPL]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < MERGE_NPL; ++i) {
        const int c = lane + 32 * i;
        if (c < C) {
            const double2 raw = __ldcg(reinterpret_cast<const double2*>(prow + c));
            q[i] = *reinterpret_cast<const Partial*>(&raw);
        } else {
            q[i].m = -INFINITY;
            q[i].amax = INT_MAX;
            q[i].z = 0.0;
        }
    }
}

// merge_row on partials already loaded by load_row.
__device__ __forceinline__ void merge_loaded(const Partial (&q)[MERGE_NPL], bool greedy, float kappa,
                                             float& M, float& Z, int& A) {
    constexpr int NPL = MERGE_NPL;
    {
        float lm = -INFINITY;
#pragma unroll
        for (int i = 0; i < NPL; ++i) lm = fmaxf(lm, q[i].m);
        M = warp_max(lm);
        A = INT_MAX;
        Z = 0.f;
        if (greedy) {
            int la = INT_MAX;
#pragma unroll
            for (int i = 0; i < NPL; ++i)
                if (q[i].m == M) la = min(la, q[i].amax);
            A = warp_min_int(la);
        } else {
            float lz = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int i = 0; i < NPL; ++i)
                    if (q[i].m != -INFINITY && q[i].z != 0.0)
                        lz = fmaf(float(q[i].z), rebase_factor(q[i].m, M, kappa), lz);
            }
            Z = warp_sum_f(lz);
        }
    }
}

__device__ __forceinline__ void merge_row(const Partial* prow, int C, bool greedy, float kappa,
                                          float& M, float& Z, int& A) {
    const int lane = threadIdx.x & 31;
    if (C <= 32 * MERGE_NPL) {
        Partial q[MERGE_NPL];
        load_row(prow, C, q);
        merge_loaded(q, greedy, kappa, M, Z, A);
    } else {  // long vocabularies: pairwise merges over the lane's chunks
        float m = -INFINITY;
        int am = INT_MAX;
        float z = 0.f;
        for (int c = lane; c < C; c += 32) {
            const double2 raw = __ldcg(reinterpret_cast<const double2*>(prow + c));
            const Partial q = *reinterpret_cast<const Partial*>(&raw);
            if (greedy)
                merge_argmax(m, am, q.m, q.amax);
            else
                merge_sum(m, z, q.m, float(q.z), kappa);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, o);
            if (greedy)
                merge_argmax(m, am, om, __shfl_xor_sync(0xffffffffu, am, o));
            else
                merge_sum(m, z, om, __shfl_xor_sync(0xffffffffu, z, o), kappa);
        }
        M = m;
        A = am;
        Z = z;
    }
}

// Steps 2-4 of request b (whole warp; lane j holds row j's merged M, Z, A for
// jlo <= j <= jhi).  n = num_draft[b], kappa = log2(e) / T (0 for greedy).
static __device__ __noinline__ void accept_decide(const Params& P, int b, int n, bool greedy,
                                                  float kappa, const AccLoads& L, float my_m,
                                                  int my_amax, float my_Z) {
    const int lane = threadIdx.x & 31;
    const int K1 = P.K1;
    int32_t* out = P.out_ids + (size_t)b * K1;
    const float NaN = __int_as_float(0x7fc00000);
    const bool ee = P.round >= 0;
    const int jlo = ee ? P.round : 0, jhi = ee ? P.round : n;
    const bool row_lane = lane >= jlo && lane <= jhi;
    const bool draft_lane = row_lane && lane < n;
    const int x = L.x;
    const float2 g = L.g;
    const uint4 rb = L.rb;
    const bool typical = P.rule == RULE_TYPICAL;

    auto fail = [&](int flags) {
        if (lane < K1) out[lane] = -1;
        if (P.dbg_rows && lane < K1) {
            float* d = P.dbg_rows + ((size_t)b * K1 + lane) * 4;
            d[0] = d[1] = d[2] = NaN;
            d[3] = -1.f;
        }
        if (lane == 0) {
            P.out_nacc[b] = -1;
            atomicOr(P.status, flags);
            if (P.dbg_req) {
                float* d = P.dbg_req + (size_t)b * 4;
                d[0] = float(MODE_BAD);
                d[1] = d[2] = d[3] = NaN;
            }
        }
    };

    // 2. validation of the draft ids and rows this request uses
    const unsigned bad_id = __ballot_sync(0xffffffffu, draft_lane && (x < 0 || x >= P.V));
    const unsigned empty = __ballot_sync(0xffffffffu, !greedy && row_lane && my_m == -INFINITY);
    if (bad_id | empty) {
        fail((bad_id ? int(SPEC_BADBIT_DRAFT_ID) : 0) | (empty ? int(SPEC_BADBIT_EMPTY_ROW) : 0));
        return;
    }

    // acceptance of draft `lane`
    bool acc = false;
    float p = NaN;
    float u = NaN;
    if (draft_lane) {
        if (greedy) {
            acc = (x == my_amax);
        } else {
            const float lx = g.x, qx = g.y;
            p = __fdiv_rn(exp2f(weight_arg(lx, my_m, offset_of(my_m, kappa), kappa)), my_Z);
            if (typical) {
                // "投机采样" 验收标准, Typical Acceptance: a hard threshold on
                // the target's probability of the draft
                acc = (p > 0.f) && (p >= P.threshold);
            } else {
                u = uniform01(rb.x);
                // u <= p / q  <=>  u q <= p (q > 0); the product of two floats
                // is exact in double, so the comparison takes no rounding
                acc = (p > 0.f) && (qx == 0.f || double(u) * double(qx) <= double(p));
            }
        }
    }

    auto write_dbg = [&]() {
        float* d = P.dbg_rows + ((size_t)b * K1 + lane) * 4;
        if (draft_lane) {
            d[0] = greedy ? NaN : p;
            d[1] = greedy ? NaN : u;
            d[2] = greedy ? NaN : float(my_Z);
            d[3] = acc ? 1.f : 0.f;
        } else {
            d[0] = d[1] = d[2] = NaN;
            d[3] = -1.f;
        }
    };

    // 3. first rejection
    const unsigned accm = __ballot_sync(0xffffffffu, acc);
    if (ee && ((accm >> jlo) & 1u)) {  // early exit: draft jlo kept, row jlo + 1 is next
        if (lane == jlo) {
            out[jlo] = x;
            const int i = atomicAdd(&P.hdr[HDR_ROUND + jlo + 1], 1);
            P.rowlist[(size_t)(jlo + 1) * P.B + i] = b * K1 + jlo + 1;
            if (P.dbg_rows) write_dbg();
        }
        return;
    }
    const int a = ee ? jlo : min(n, __ffs(~accm) - 1);

    // 4. outputs (early exit wrote the kept drafts round by round)
    if (lane < a) {
        if (!ee) out[lane] = x;
    } else if (lane > a && lane < K1) {
        out[lane] = -1;
    }
    if (greedy && lane == a) out[a] = my_amax;
    if (lane == 0) P.out_nacc[b] = a;
    if (!greedy && lane == a) {
        ReqRec r;
        // typical acceptance draws the next token from p at row a, refused
        // draft or not: it joins the bonus queue
        const bool resid = a < n && !typical;
        r.mode = typical ? MODE_TYPICAL : (resid ? MODE_RESIDUAL : MODE_BONUS);
        r.erow = a;
        r.m = my_m;
        r.kappa = kappa;
        r.Z = double(my_Z);
        r.u2 = uniform01(rb.y);
        r.b = b;
        if (resid) {
            const int i = atomicAdd(&P.hdr[HDR_NRES], 1);
            P.res_rec[i] = r;
        } else {
            const int i = atomicAdd(&P.hdr[HDR_NBONUS], 1);
            P.bonus_rec[i] = r;
        }
    }
    if (P.dbg_rows && lane < K1 && lane >= jlo) write_dbg();
    if (P.dbg_req && greedy && lane == 0) {
        float* d = P.dbg_req + (size_t)b * 4;
        d[0] = float(MODE_GREEDY);
        d[1] = float(a);
        d[2] = d[3] = NaN;
    }
}

// Request b in an early-exit pass (valid: k_plan has checked num_draft and
// temperature); whole warp.  n and kappa come from the caller, which already
// holds them.
static __device__ __noinline__ void accept_request(const Params& P, int b, int n, bool greedy,
                                                   float kappa) {
    const int lane = threadIdx.x & 31;
    const bool ee = P.round >= 0;
    const int jlo = ee ? P.round : 0, jhi = ee ? P.round : n;
    const AccLoads L = accept_loads(P, b, n, greedy, jlo, jhi);
    float my_m = -INFINITY, my_Z = 0.f;
    int my_amax = INT_MAX;
    const Partial* pb = P.part + (size_t)b * P.K1 * P.C;
    for (int j = jlo; j <= jhi; ++j) {
        float M, Z;
        int A;
        merge_row(pb + (size_t)j * P.C, P.C, greedy, kappa, M, Z, A);
        if (lane == j) {
            my_m = M;
            my_amax = A;
            my_Z = Z;
        }
    }
    accept_decide(P, b, n, greedy, kappa, L, my_m, my_amax, my_Z);
}

}  // namespace sv
