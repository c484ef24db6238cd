// accept.cu -- k_accept: one warp per request.
//
// Lane j owns row j of the request.  Steps (pages cited by title / section):
//   1. merge the chunk partials of every row j <= n_b into the row's max m_j,
//      normaliser Z_j = sum_x 2^((l_j(x) - m_j) kappa) (float64) and, for
//      greedy rows, the lowest-index argmax;
//   2. acceptance of draft x_j ("深入推测解码" 保证原始分布 step 3,
//      "RTP-LLM Speculative Engine" 拒绝采样算法): p = 2^((l_j(x_j) - m_j) kappa)
//      / Z_j in float64, u_j = Philox lane 0 of row j, accept iff p > 0 and
//      (q_j(x_j) == 0 or u_j <= p / q_j(x_j)); greedy ("投机采样" 精确匹配):
//      accept iff x_j is the row's argmax;
//   3. first-reject scan in-warp: a_b = position of the lowest zero of the
//      ballot of acceptance bits ("投机采样" 第五步: drafts after a rejected
//      one are discarded);
//   4. write the accepted prefix and the -1 tail; greedy requests also write
//      the emitted token (argmax of row a_b); sampling requests are queued for
//      k_sample (residual at row a_b < n_b, bonus at row a_b == n_b).
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace sv {

namespace {

// (m, z) <- (m, z) (+) (m2, z2): sums of 2^((l - m) kappa) with different maxima.
__device__ __forceinline__ void merge_sum(float& m, double& z, float m2, double z2, float kappa) {
    if (m2 > m) {
        const float tm = m;
        m = m2;
        m2 = tm;
        const double tz = z;
        z = z2;
        z2 = tz;
    }
    if (m2 != -INFINITY && z2 != 0.0) z += z2 * exp2(double(__fmul_rn(__fsub_rn(m2, m), kappa)));
}

__device__ __forceinline__ void merge_argmax(float& m, int& a, float m2, int a2) {
    if (m2 > m || (m2 == m && a2 < a)) {
        m = m2;
        a = a2;
    }
}

}  // namespace

__global__ void __launch_bounds__(ACCEPT_WARPS * 32) k_accept(Params P) {
    griddep_launch_dependents();
    griddep_wait();  // partials of k_row_stats (and, transitively, k_plan)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x * ACCEPT_WARPS + warp;
    if (b >= P.B) return;
    const int K1 = P.K1;
    int32_t* out = P.out_ids + (size_t)b * K1;
    const float NaN = __int_as_float(0x7fc00000);

    auto fail = [&](int flags) {
        if (lane < K1) out[lane] = -1;
        if (P.dbg_rows && lane < K1) {
            float* d = P.dbg_rows + ((size_t)b * K1 + lane) * 4;
            d[0] = d[1] = d[2] = NaN;
            d[3] = -1.f;
        }
        if (lane == 0) {
            P.out_nacc[b] = -1;
            P.reqs[b].mode = MODE_BAD;
            atomicOr(P.status, flags);
            if (P.dbg_req) {
                float* d = P.dbg_req + (size_t)b * 4;
                d[0] = float(MODE_BAD);
                d[1] = d[2] = d[3] = NaN;
            }
        }
    };

    const int flags0 = P.req_flags[b];
    if (flags0) {
        fail(flags0);
        return;
    }
    const int n = P.num_draft[b];
    const float T = P.temp[b];
    const bool greedy = (T == 0.f);
    const float kappa = greedy ? 0.f : kappa_of(T);

    // 1. per-row merge; lane j keeps row j
    float my_m = -INFINITY;
    int my_amax = INT_MAX;
    double my_Z = 0.0;
    for (int j = 0; j <= n; ++j) {
        const Partial* pr = P.part + ((size_t)b * K1 + j) * P.C;
        float m = -INFINITY;
        int am = INT_MAX;
        double z = 0.0;
        for (int c = lane; c < P.C; c += 32) {
            const Partial q = pr[c];
            if (greedy)
                merge_argmax(m, am, q.m, q.amax);
            else
                merge_sum(m, z, q.m, q.z, kappa);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, o);
            if (greedy) {
                merge_argmax(m, am, om, __shfl_xor_sync(0xffffffffu, am, o));
            } else {
                merge_sum(m, z, om, __shfl_xor_sync(0xffffffffu, z, o), kappa);
            }
        }
        if (lane == j) {
            my_m = m;
            my_amax = am;
            my_Z = z;
        }
    }

    // 2. validation of the draft ids and rows this request uses
    const bool draft_lane = lane < n;
    const int x = draft_lane ? P.ids[(size_t)b * P.K + lane] : -1;
    const unsigned bad_id = __ballot_sync(0xffffffffu, draft_lane && (x < 0 || x >= P.V));
    const unsigned empty = __ballot_sync(0xffffffffu, !greedy && lane <= n && my_m == -INFINITY);
    if (bad_id | empty) {
        fail((bad_id ? int(SPEC_BADBIT_DRAFT_ID) : 0) | (empty ? int(SPEC_BADBIT_EMPTY_ROW) : 0));
        return;
    }

    // acceptance of draft `lane`
    bool acc = false;
    double p = NaN;
    float u = NaN;
    uint4 rb = make_uint4(0, 0, 0, 0);
    if (!greedy && lane <= n) rb = row_block(P, b, lane);
    if (draft_lane) {
        if (greedy) {
            acc = (x == my_amax);
        } else {
            const float lx = load_logit(P.logits, P.dtype, ((size_t)b * K1 + lane) * P.V + x);
            const float qx = __ldg(P.probs + ((size_t)b * P.K + lane) * P.V + x);
            p = exp2(double(__fmul_rn(__fsub_rn(lx, my_m), kappa))) / my_Z;
            u = uniform01(rb.x);
            acc = (p > 0.0) && (qx == 0.f || double(u) <= p / double(qx));
        }
    }

    // 3. first rejection
    const unsigned accm = __ballot_sync(0xffffffffu, acc);
    const int a = min(n, __ffs(~accm) - 1);

    // 4. outputs
    if (lane < a)
        out[lane] = x;
    else if (lane > a && lane < K1)
        out[lane] = -1;
    if (greedy && lane == a) out[a] = my_amax;
    if (lane == 0) P.out_nacc[b] = a;
    if (!greedy && lane == a) {
        ReqRec r;
        r.mode = a < n ? MODE_RESIDUAL : MODE_BONUS;
        r.erow = a;
        r.m = my_m;
        r.kappa = kappa;
        r.Z = my_Z;
        r.u2 = uniform01(rb.y);
        r.b = b;
        P.reqs[b] = r;
        if (a < n) {
            const int i = atomicAdd(&P.hdr[HDR_NRES], 1);
            P.res_list[i] = b;
            P.res_cnt[i] = 0;
        } else {
            const int i = atomicAdd(&P.hdr[HDR_NBONUS], 1);
            P.bonus_list[i] = b;
        }
    }
    if (P.dbg_rows && lane < K1) {
        float* d = P.dbg_rows + ((size_t)b * K1 + lane) * 4;
        if (draft_lane) {
            d[0] = greedy ? NaN : float(p);
            d[1] = greedy ? NaN : u;
            d[2] = greedy ? NaN : float(my_Z);
            d[3] = acc ? 1.f : 0.f;
        } else {
            d[0] = d[1] = d[2] = NaN;
            d[3] = -1.f;
        }
    }
    if (P.dbg_req && greedy && lane == 0) {
        float* d = P.dbg_req + (size_t)b * 4;
        d[0] = float(MODE_GREEDY);
        d[1] = float(a);
        d[2] = d[3] = NaN;
    }
}

}  // namespace sv
