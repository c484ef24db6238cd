// plan.cu -- k_plan: validate the per-request scalars and compact the rows the
// verifier must read.
//
// Request b needs rows j = 0..n_b of its target logits: rows 0..n_b-1 for the
// acceptance tests of its drafts and row n_b for the bonus token ("投机采样",
// 第二步: one target pass yields p_1..p_{gamma+1}).  Requests with a bad
// num_draft or temperature contribute no rows and are flagged.
#include <cfloat>

#include "common.cuh"

namespace sv {

__global__ void __launch_bounds__(PLAN_THREADS) k_plan(Params P) {
    __shared__ int warp_excl[PLAN_THREADS / 32];
    __shared__ int carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    griddep_launch_dependents();
    if (tid < SPEC_MAX_K + 1) P.hdr[HDR_ROUND + tid] = 0;
    if (tid == 0) {
        P.hdr[HDR_NRES] = 0;
        P.hdr[HDR_NBONUS] = 0;
        P.hdr[HDR_CLAIM] = 0;
        *P.status = 0;
        carry = 0;
    }
    __syncthreads();
    int flags_any = 0;
    for (int base = 0; base < P.B; base += PLAN_THREADS) {
        const int b = base + tid;
        int rows = 0;
        if (b < P.B) {
            const int n = P.num_draft[b];
            const float T = P.temp[b];
            int flags = 0;
            if (n < 0 || n > P.K) flags |= SPEC_BADBIT_NUM_DRAFT;
            if (!(T >= 0.f) || T > FLT_MAX) flags |= SPEC_BADBIT_TEMPERATURE;
            if (P.tree) {  // n counts the nodes, the root included
                flags = 0;
                if (n < 1 || n > P.K1) flags |= SPEC_BADBIT_NUM_DRAFT;
                if (!(T >= 0.f) || T > FLT_MAX) flags |= SPEC_BADBIT_TEMPERATURE;
                if (!flags && T > 0.f && n > 1 && P.probs == nullptr)
                    flags |= SPEC_BADBIT_NO_PROBS;
            } else if (!flags && T > 0.f && n > 0 && P.probs == nullptr &&
                       P.rule == RULE_LOSSLESS) {
                flags |= SPEC_BADBIT_NO_PROBS;
            }
            if (!flags && P.round == 0)  // early exit: every draft id is checked up front
                for (int j = 0; j < n; ++j) {
                    const int x = P.ids[(size_t)b * P.K + j];
                    if (x < 0 || x >= P.V) flags |= SPEC_BADBIT_DRAFT_ID;
                }
            // early exit starts with row 0 of every request
            rows = flags ? 0 : (P.tree ? n : (P.round == 0 ? 1 : n + 1));
            P.req_flags[b] = flags;
            P.cnt[b] = 0;
            flags_any |= flags;
            if (flags) {  // no row of a bad request is read: its outputs are final here
                for (int j = 0; j < P.K1; ++j) P.out_ids[(size_t)b * P.K1 + j] = -1;
                P.out_nacc[b] = -1;
                if (P.out_last) P.out_last[b] = -1;
                const float NaN = __int_as_float(0x7fc00000);
                if (P.dbg_rows)
                    for (int j = 0; j < P.K1; ++j) {
                        float* d = P.dbg_rows + ((size_t)b * P.K1 + j) * 4;
                        d[0] = d[1] = d[2] = NaN;
                        d[3] = -1.f;
                    }
                if (P.dbg_req) {
                    float* d = P.dbg_req + (size_t)b * 4;
                    d[0] = float(MODE_BAD);
                    d[1] = d[2] = d[3] = NaN;
                }
            }
        }
        // block-wide exclusive scan of the row counts
        int incl = rows;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) warp_excl[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int tot = warp_excl[lane];
            int s = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += v;
            }
            warp_excl[lane] = s - tot;
        }
        __syncthreads();
        const int start = carry + warp_excl[warp] + incl - rows;
        for (int j = 0; j < rows; ++j) P.rowlist[start + j] = b * P.K1 + j;
        __syncthreads();
        if (tid == PLAN_THREADS - 1) carry = start + rows;
        __syncthreads();
    }
    if (flags_any) atomicOr(P.status, flags_any);
    if (tid == 0) P.hdr[HDR_ROWS] = carry;
}

}  // namespace sv
