// tree.cu -- k_tree_walk: token-tree verification, one CTA per request.
//
// The drafts of a request form a trie ("投机采样", 验证方案: candidate
// sequences that share a prefix share a node; the target scores every node
// in one pass).  Node 0 is the accepted context, node c >= 1 carries a draft
// token and its parent (an earlier node); row v of the target logits is the
// target's distribution of the token that follows node v, row c of the draft
// probabilities the distribution node c's token was drawn from.  k_row_stats
// has reduced every node row to per-chunk (max, sum, argmax) partials; this
// kernel merges them, checks the trie and walks it from the root:
//   greedy rows ("投机采样" 精确匹配): at node v the first child (in index
//     order) whose token is the argmax of row v is kept; otherwise the argmax
//     is the emitted token;
//   sampling rows: the children of v are tested in index order against a
//     running target r, r = p_v first ("深入推测解码" 保证原始分布 step 3
//     applied to each sibling): child c is kept with probability
//     min(1, r(x_c) / q_c(x_c)); after a rejection r becomes
//     norm(max(0, r - q_c)) (step 4; kept as it was if that has no mass).
//     When no child is kept the token is drawn from the last residual (from r
//     if it had no mass, from p_v at a node without children) by the inverse
//     CDF with the emission uniform of node v.
// Uniforms: child c's acceptance uniform is Philox lane 0 of row c - 1, node
// v's emission uniform lane 1 of row v, so that a trie with one child per
// node is verified exactly like a chain of drafts.
// Each normaliser of a residual is one CTA-wide pass over the vocabulary
// (the node's logits row and the q rows of the siblings rejected so far),
// which also leaves the per-chunk masses that the inverse CDF needs.
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace sv {

namespace {

constexpr int TW = TREE_THREADS / 32;  // warps per CTA
constexpr int GROUPS = TILE / 8 / 32;  // 8-token groups per lane in a chunk
#ifndef SV_TREE_BATCH
#define SV_TREE_BATCH 4
#endif
constexpr int PASS_BATCH = SV_TREE_BATCH;  // groups of a pass whose loads are issued together
static_assert(GROUPS % PASS_BATCH == 0, "whole batches of groups per chunk");

template <int DT>
__device__ __forceinline__ void logits8(const Params& P, size_t row_base, int y0, float (&l)[8]) {
    if constexpr (DT == SPEC_BF16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(
            reinterpret_cast<const uint16_t*>(P.logits) + row_base + y0));
        l[0] = bf16_lo(v.x); l[1] = bf16_hi(v.x);
        l[2] = bf16_lo(v.y); l[3] = bf16_hi(v.y);
        l[4] = bf16_lo(v.z); l[5] = bf16_hi(v.z);
        l[6] = bf16_lo(v.w); l[7] = bf16_hi(v.w);
    } else {
        const float4* s = reinterpret_cast<const float4*>(
            reinterpret_cast<const float*>(P.logits) + row_base + y0);
        const float4 a = __ldg(s), c = __ldg(s + 1);
        l[0] = a.x; l[1] = a.y; l[2] = a.z; l[3] = a.w;
        l[4] = c.x; l[5] = c.y; l[6] = c.z; l[7] = c.w;
    }
}
__device__ __forceinline__ void probs8(const float* row, int y0, float (&q)[8]) {
    const float4* s = reinterpret_cast<const float4*>(row + y0);
    const float4 a = __ldg(s), c = __ldg(s + 1);
    q[0] = a.x; q[1] = a.y; q[2] = a.z; q[3] = a.w;
    q[4] = c.x; q[5] = c.y; q[6] = c.z; q[7] = c.w;
}

// The running target and its residuals: r_0 = p_v and, for each rejected
// sibling e with a residual of positive mass, r_e = max(0, r_{e-1} - q_e) / S_e.
struct Chain {
    int n;                          // subtractions so far
    int child[TREE_MAX_NODES];      // their nodes
    float inv[TREE_MAX_NODES];      // float(1 / S_e)
};

// float32 value of r_k at the 8 tokens of a group (w: max(0, r_{k-1} - q)
// before the last normalisation when `last_raw`), the same operations at
// every use so that a token's weight is identical in every pass.
__device__ __forceinline__ void chain8(const float (&p)[8], const Chain& ch, int k,
                                       const float* const* qrows, int y0, float (&r)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = p[e];
    for (int i = 0; i < k; ++i) {
        float q[8];
        probs8(qrows[i], y0, q);
#pragma unroll
        for (int e = 0; e < 8; ++e) r[e] = __fmul_rn(fmaxf(__fsub_rn(r[e], q[e]), 0.f), ch.inv[i]);
    }
}

}  // namespace

template <int DT>
__device__ __forceinline__ void tree_walk_body(const Params& P) {
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int N = P.K1;
    if (b >= P.B || P.req_flags[b] != 0) return;  // bad requests: k_plan wrote their outputs
    __shared__ int s_par[TREE_MAX_NODES], s_tok[TREE_MAX_NODES], s_amax[TREE_MAX_NODES];
    __shared__ float s_m[TREE_MAX_NODES], s_z[TREE_MAX_NODES];
    __shared__ Chain s_ch;
    __shared__ const float* s_qrows[TREE_MAX_NODES + 1];
    __shared__ double s_red[TW];
    __shared__ int s_flag;
    const int n = P.num_draft[b];
    const float T = P.temp[b];
    const bool greedy = (T == 0.f);
    const float kappa = greedy ? 0.f : kappa_of(T);
    const float NaN = __int_as_float(0x7fc00000);
    int32_t* out = P.out_ids + (size_t)b * N;

    // the trie
    if (tid < TREE_MAX_NODES) {
        s_par[tid] = (tid >= 1 && tid < n) ? P.parents[(size_t)b * N + tid] : -1;
        s_tok[tid] = (tid >= 1 && tid < n) ? P.ids[(size_t)b * N + tid] : -1;
    }
    if (tid == 0) s_flag = 0;
    __syncthreads();
    if (tid >= 1 && tid < n) {
        int f = 0;
        if (s_par[tid] < 0 || s_par[tid] >= tid) f |= SPEC_BADBIT_TREE;
        if (s_tok[tid] < 0 || s_tok[tid] >= P.V) f |= SPEC_BADBIT_DRAFT_ID;
        if (f) atomicOr(&s_flag, f);
    }
    // merge the chunk partials of every node row: warp w takes rows w, w + TW, ...
    const Partial* pb = P.part + (size_t)b * N * P.C;
    for (int v = warp; v < n; v += TW) {
        float m = -INFINITY, z = 0.f;
        int am = INT_MAX;
        for (int c = lane; c < P.C; c += 32) {
            const Partial q = pb[(size_t)v * P.C + c];
            if (greedy) {
                if (q.m > m || (q.m == m && q.amax < am)) {
                    m = q.m;
                    am = q.amax;
                }
            } else if (q.m != -INFINITY && q.z != 0.0) {
                const float zc = float(q.z);
                if (q.m > m) {
                    if (m != -INFINITY && z != 0.f) z = __fmul_rn(z, rebase_factor(m, q.m, kappa));
                    m = q.m;
                    z = __fadd_rn(z, zc);
                } else {
                    z = fmaf(zc, rebase_factor(q.m, m, kappa), z);
                }
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float om = __shfl_xor_sync(0xffffffffu, m, o);
            const float oz = __shfl_xor_sync(0xffffffffu, z, o);
            const int oa = __shfl_xor_sync(0xffffffffu, am, o);
            if (greedy) {
                if (om > m || (om == m && oa < am)) {
                    m = om;
                    am = oa;
                }
            } else if (om != -INFINITY && oz != 0.f) {
                if (om > m) {
                    if (m != -INFINITY && z != 0.f) z = __fmul_rn(z, rebase_factor(m, om, kappa));
                    m = om;
                    z = __fadd_rn(z, oz);
                } else {
                    z = fmaf(oz, rebase_factor(om, m, kappa), z);
                }
            }
        }
        if (lane == 0) {
            s_m[v] = m;
            s_z[v] = z;
            s_amax[v] = am;
            if (!greedy && m == -INFINITY) atomicOr(&s_flag, int(SPEC_BADBIT_EMPTY_ROW));
        }
    }
    __syncthreads();
    if (s_flag) {
        if (tid < N) out[tid] = -1;
        if (tid == 0) {
            P.out_nacc[b] = -1;
            P.out_last[b] = -1;
            atomicOr(P.status, s_flag);
            if (P.dbg_req) {
                float* d = P.dbg_req + (size_t)b * 4;
                d[0] = float(MODE_BAD);
                d[1] = d[2] = d[3] = NaN;
            }
        }
        if (P.dbg_rows && tid < N) {
            float* d = P.dbg_rows + ((size_t)b * N + tid) * 4;
            d[0] = d[1] = d[2] = NaN;
            d[3] = -1.f;
        }
        return;
    }
    if (P.dbg_rows && tid < N) {
        float* d = P.dbg_rows + ((size_t)b * N + tid) * 4;
        d[0] = d[1] = d[2] = NaN;
        d[3] = -1.f;
    }

    // the walk (every thread follows the same decisions, read from shared memory)
    __shared__ int s_v, s_depth, s_next, s_child, s_mode;
    __shared__ float s_u2, s_total_f;
    __shared__ double s_total;
    if (tid == 0) {
        s_v = 0;
        s_depth = 0;
    }
    __syncthreads();
    for (;;) {
        const int v = s_v;
        const size_t vbase = ((size_t)b * N + v) * P.V;
        if (greedy) {
            if (tid == 0) {
                const int g = s_amax[v];
                int next = -1;
                for (int c = v + 1; c < n && next < 0; ++c)
                    if (s_par[c] == v) {
                        if (P.dbg_rows) P.dbg_rows[((size_t)b * N + c) * 4 + 3] = s_tok[c] == g;
                        if (s_tok[c] == g) next = c;
                    }
                if (next >= 0) {
                    out[s_depth++] = s_tok[next];
                    s_v = next;
                } else {
                    out[s_depth] = g;
                    s_next = -2;  // done
                }
                if (next >= 0) s_next = next;
            }
            __syncthreads();
            if (s_next == -2) break;
            continue;
        }
        // sampling: the children of v against the running target
        const float m = s_m[v], cv = offset_of(m, kappa), invZ = float(1.0 / double(s_z[v]));
        if (tid == 0) {
            s_ch.n = 0;
            s_qrows[0] = nullptr;
            s_next = -1;
            s_mode = MODE_BONUS;
        }
        __syncthreads();
        bool accepted = false;
        for (int c = v + 1; c < n; ++c) {
            if (s_par[c] != v) continue;
            // the acceptance test of child c (thread 0)
            if (tid == 0) {
                const int x = s_tok[c];
                const int x0 = x & ~7;
                float l[8], p[8], r[8];
                logits8<DT>(P, vbase, x0, l);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    p[e] = __fmul_rn(ex2_approx(weight_arg(l[e], m, cv, kappa)), invZ);
                chain8(p, s_ch, s_ch.n, s_qrows, x0, r);
                const float rx = r[x - x0];
                const float qx = __ldg(P.probs + ((size_t)b * N + c) * P.V + x);
                const float u = uniform01(row_block(P, b, c - 1).x);
                const bool acc = rx > 0.f && (qx == 0.f || double(u) * double(qx) <= double(rx));
                if (P.dbg_rows) {
                    float* d = P.dbg_rows + ((size_t)b * N + c) * 4;
                    d[0] = rx;
                    d[1] = u;
                    d[2] = qx;
                    d[3] = acc ? 1.f : 0.f;
                }
                s_child = c;
                if (acc) {
                    out[s_depth++] = x;
                    s_v = c;
                    s_next = c;
                }
                s_qrows[s_ch.n] = P.probs + ((size_t)b * N + c) * P.V;  // candidate subtraction
            }
            __syncthreads();
            if (s_next >= 0) {
                accepted = true;
                break;
            }
            // rejected: S = sum_y max(0, r_k(y) - q_c(y)), and its chunk masses
            const int k = s_ch.n;
            double part = 0.0;
            for (int ch = warp; ch < P.C && k == 0; ch += TW) {
                // first rejection at this node: r = p, so each group needs its
                // logits and one q row; PASS_BATCH groups' loads are issued
                // before their arithmetic (same operations, same order)
                const int y_end = min(TILE, P.V - ch * TILE);
                const float* qrow = s_qrows[0];
                float acc_f = 0.f;
#pragma unroll 1
                for (int g0 = 0; g0 < GROUPS; g0 += PASS_BATCH) {
                    float l[PASS_BATCH][8], q[PASS_BATCH][8];
#pragma unroll
                    for (int u = 0; u < PASS_BATCH; ++u) {
                        const int gl = (g0 + u) * 32 + lane;
                        if (gl * 8 < y_end) {
                            logits8<DT>(P, vbase, ch * TILE + gl * 8, l[u]);
                            probs8(qrow, ch * TILE + gl * 8, q[u]);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < PASS_BATCH; ++u) {
                        const int gl = (g0 + u) * 32 + lane;
                        if (gl * 8 >= y_end) continue;
                        float r[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float pe = __fmul_rn(ex2_approx(weight_arg(l[u][e], m, cv, kappa)), invZ);
                            r[e] = fmaxf(__fsub_rn(pe, q[u][e]), 0.f);
                        }
#pragma unroll
                        for (int h = 4; h; h >>= 1)
#pragma unroll
                            for (int e = 0; e < h; ++e) r[e] = __fadd_rn(r[e], r[e + h]);
                        acc_f = __fadd_rn(acc_f, r[0]);
                    }
                }
                const float cm = warp_sum_f(acc_f);
                if (lane == 0) P.tmass[(size_t)b * P.C + ch] = cm;
                part += double(cm);
            }
            for (int ch = warp; ch < P.C && k > 0; ch += TW) {
                const int y_end = min(TILE, P.V - ch * TILE);
                float acc_f = 0.f;
#pragma unroll 1
                for (int g = 0; g < GROUPS; ++g) {
                    const int y0 = ch * TILE + (g * 32 + lane) * 8;
                    if ((g * 32 + lane) * 8 >= y_end) continue;
                    float l[8], p[8], r[8], q[8];
                    logits8<DT>(P, vbase, y0, l);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        p[e] = __fmul_rn(ex2_approx(weight_arg(l[e], m, cv, kappa)), invZ);
                    chain8(p, s_ch, k, s_qrows, y0, r);
                    probs8(s_qrows[k], y0, q);
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = fmaxf(__fsub_rn(r[e], q[e]), 0.f);
#pragma unroll
                    for (int h = 4; h; h >>= 1)
#pragma unroll
                        for (int e = 0; e < h; ++e) r[e] = __fadd_rn(r[e], r[e + h]);
                    acc_f = __fadd_rn(acc_f, r[0]);
                }
                const float cm = warp_sum_f(acc_f);
                if (lane == 0) P.tmass[(size_t)b * P.C + ch] = cm;
                part += double(cm);
            }
            if (lane == 0) s_red[warp] = part;
            __syncthreads();
            if (tid == 0) {
                double S = 0.0;
                for (int w = 0; w < TW; ++w) S += s_red[w];
                if (S > 0.0) {  // the residual becomes the running target
                    s_ch.child[k] = s_child;
                    s_ch.inv[k] = float(1.0 / S);
                    s_ch.n = k + 1;
                    s_mode = MODE_RESIDUAL;
                    s_total = S;
                } else {
                    s_mode = MODE_FALLBACK;  // no mass: r stays
                }
            }
            __syncthreads();
        }
        if (accepted) continue;

        // no child kept: draw from the weights of the last step
        //   bonus (no children):   p_v, chunk masses summed here
        //   residual:              max(0, r_{k-1} - q_last) = r_k * S_k, masses of the last pass
        //   fallback (no mass):    r_k, chunk masses summed here
        const int mode = s_mode;
        const int kk = s_ch.n;
        const bool resid_w = (mode == MODE_RESIDUAL);
        if (!resid_w) {
            double part = 0.0;
            for (int ch = warp; ch < P.C; ch += TW) {
                const int y_end = min(TILE, P.V - ch * TILE);
                float acc_f = 0.f;
#pragma unroll 1
                for (int g = 0; g < GROUPS; ++g) {
                    const int y0 = ch * TILE + (g * 32 + lane) * 8;
                    if ((g * 32 + lane) * 8 >= y_end) continue;
                    float l[8], p[8], r[8];
                    logits8<DT>(P, vbase, y0, l);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        p[e] = __fmul_rn(ex2_approx(weight_arg(l[e], m, cv, kappa)), invZ);
                    chain8(p, s_ch, kk, s_qrows, y0, r);
#pragma unroll
                    for (int h = 4; h; h >>= 1)
#pragma unroll
                        for (int e = 0; e < h; ++e) r[e] = __fadd_rn(r[e], r[e + h]);
                    acc_f = __fadd_rn(acc_f, r[0]);
                }
                const float cm = warp_sum_f(acc_f);
                if (lane == 0) P.tmass[(size_t)b * P.C + ch] = cm;
                part += double(cm);
            }
            if (lane == 0) s_red[warp] = part;
        }
        __syncthreads();
        if (warp == 0) {
            // level 1: the chunk holding u' * total, chunk masses in chunk order
            const float u2 = uniform01(row_block(P, b, v).y);
            double total = 0.0;
            for (int c0 = 0; c0 < P.C; c0 += 32)
                total += warp_sum(c0 + lane < P.C ? double(P.tmass[(size_t)b * P.C + c0 + lane])
                                                 : 0.0);
            const double t = double(u2) * total;
            int chosen = -1;
            double before = 0.0, carry = 0.0;
            for (int c0 = 0; c0 < P.C && chosen < 0; c0 += 32) {
                const double mc = c0 + lane < P.C ? double(P.tmass[(size_t)b * P.C + c0 + lane]) : 0.0;
                double incl = mc;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const double y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                incl += carry;
                const unsigned hit = __ballot_sync(0xffffffffu, incl >= t && mc > 0.0);
                if (hit) {
                    const int l = __ffs(hit) - 1;
                    chosen = c0 + l;
                    before = __shfl_sync(0xffffffffu, incl - mc, l);
                }
                carry = __shfl_sync(0xffffffffu, incl, 31);
            }
            int x = 0;
            if (chosen >= 0) {
                // level 2: the chunk's weights in token order (8-token groups)
                const float tloc = float(t - before);
                const int c0 = chosen * TILE, nel = min(TILE, P.V - c0);
                const float* qlast = resid_w ? s_qrows[kk - 1] : nullptr;
                auto weight8 = [&](int g, float (&w)[8]) {
                    const int y0 = c0 + g * 8;
                    float l[8], p[8];
                    logits8<DT>(P, vbase, y0, l);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        p[e] = __fmul_rn(ex2_approx(weight_arg(l[e], m, cv, kappa)), invZ);
                    if (resid_w) {  // max(0, r_{k-1} - q_last), as summed in the pass
                        float q[8];
                        chain8(p, s_ch, kk - 1, s_qrows, y0, w);
                        probs8(qlast, y0, q);
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[e] = fmaxf(__fsub_rn(w[e], q[e]), 0.f);
                    } else {
                        chain8(p, s_ch, kk, s_qrows, y0, w);
                    }
                };
                // block k by block k: group sums, their scan carried from the
                // blocks before, and a stop at the first block reaching tloc
                float carry_f = 0.f, bef = 0.f;
                int found = -1, glast_all = -1;
#pragma unroll 1
                for (int k = 0; k < GROUPS; ++k) {
                    const int g = k * 32 + lane;
                    float gs = 0.f;
                    if (g * 8 < nel) {
                        float w[8];
                        weight8(g, w);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            gs = __fadd_rn(gs, w[e]);
                            if (w[e] > 0.f) glast_all = g * 8 + e;
                        }
                    }
                    float incl = gs;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl = __fadd_rn(incl, y);
                    }
                    incl = __fadd_rn(carry_f, incl);
                    const unsigned hit = __ballot_sync(0xffffffffu, incl >= tloc && gs > 0.f);
                    if (hit) {
                        const int l = __ffs(hit) - 1;
                        found = k * 32 + l;
                        bef = __shfl_sync(0xffffffffu, __fsub_rn(incl, gs), l);
                        break;
                    }
                    carry_f = __shfl_sync(0xffffffffu, incl, 31);
                }
                int xl = -1;
                if (found >= 0) {
                    if (lane == (found & 31)) {
                        float w[8];
                        weight8(found, w);
                        float run = bef;
                        int lastpos = -1;
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            run = __fadd_rn(run, w[e]);
                            if (w[e] > 0.f) {
                                lastpos = found * 8 + e;
                                if (xl < 0 && run >= tloc) xl = found * 8 + e;
                            }
                        }
                        if (xl < 0) xl = lastpos;
                    }
                    xl = __shfl_sync(0xffffffffu, xl, found & 31);
                } else {
                    xl = warp_max_int(glast_all);
                }
                x = c0 + (xl < 0 ? 0 : xl);
            }
            if (lane == 0) {
                out[s_depth] = x;
                s_u2 = u2;
                s_total_f = float(total);
            }
        }
        __syncthreads();
        break;
    }
    // outputs: the path, the emitted token, -1 after
    if (tid == 0) {
        const int a = s_depth;
        for (int j = a + 1; j < N; ++j) out[j] = -1;
        P.out_nacc[b] = a;
        P.out_last[b] = s_v;
        if (P.dbg_req) {
            float* d = P.dbg_req + (size_t)b * 4;
            d[0] = float(greedy ? MODE_GREEDY : s_mode);
            d[1] = float(s_v);
            d[2] = greedy ? NaN : s_total_f;
            d[3] = greedy ? NaN : s_u2;
        }
    }
}

__global__ void __launch_bounds__(TREE_THREADS) k_tree_walk_f32(Params P) {
    tree_walk_body<SPEC_F32>(P);
}
__global__ void __launch_bounds__(TREE_THREADS) k_tree_walk_bf16(Params P) {
    tree_walk_body<SPEC_BF16>(P);
}

}  // namespace sv
