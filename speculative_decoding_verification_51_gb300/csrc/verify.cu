// verify.cu -- the verification of a batch in one persistent kernel: each
// CTA takes whole requests and verifies each one the way the pages' loop does
// ("RTP-LLM Speculative Engine" 拒绝采样算法: test draft j, stop at the first
// rejection; "深入推测解码" 伪代码: break at the first mismatch), so a request's
// rows are read only up to its first rejection, and the rejected row is read
// again for the residual while it is still in L2.
//
// Work of a CTA (one per SM, 1 request at a time, the next one claimed as the
// current one reaches its last stage):
//   prep warp     claims a request (one atomic on a counter k_prep cleared,
//                 in the order k_prep wrote: most drafts first), loads its
//                 scalars, draft tokens, q_j(x_j) and Philox uniforms, and
//                 hands the record to the decider through shared memory;
//   stream warps  (16 for bf16 logits, 8 for float32) run a sequence of
//                 passes the decider publishes: a ROW pass streams one logits
//                 row (each warp the 2048-token tiles c = w, w + NW, ...,
//                 through its own 3-slot ring of 1-D bulk copies) and leaves
//                 one Partial per tile (stats.cuh); a RESID pass streams the
//                 rejected row's logits and q_e tile by tile and leaves the
//                 tile masses of max(0, p - q);
//   decider warp  merges a finished ROW pass into (max, Z, argmax) and runs
//                 the acceptance of that row ("深入推测解码" 保证原始分布 step 3,
//                 "投机采样" 精确匹配 for greedy requests); it then publishes
//                 the next row, the residual pass, or draws the emitted token
//                 (draw.cuh: bonus from p_{n_b}, residual from the RESID
//                 masses) and writes the outputs.
// Every wait is bounded: a wait that runs out sets SPEC_BADBIT_TIMEOUT and an
// abort flag that every warp checks; stream warps then wait (bounded) for their
// copies in flight and every warp returns.
#include <cfloat>
#include <climits>

#include "accept.cuh"
#include "common.cuh"
#include "draw.cuh"
#include "stats.cuh"

namespace sv {

namespace {

constexpr int VREQ = 2;        // request records per CTA (the current one and the next)
constexpr int VBUF = 2 * VREQ; // pass result buffers: two per request record
constexpr int VDRING = 4;      // pass descriptors in flight
constexpr uint64_t VWAIT_NS = 2000000000ull;  // 2 s per bounded wait

enum { PASS_ROW = 0, PASS_RESID = 1, PASS_END = 2 };
enum { REQ_EMPTY = 0, REQ_READY = 1, REQ_ACTIVE = 2 };

template <int DT>
struct VCfg {
    static constexpr int ESZ = DT == SPEC_BF16 ? 2 : 4;
    static constexpr int NW = DT == SPEC_BF16 ? 16 : 8;  // stream warps
    static constexpr int SLOT = TILE * ESZ;               // one logits tile
    static constexpr int NSLOT = 3;                       // slots of a warp's ring
    static constexpr int QSLOTS = TILE * 4 / SLOT;        // slots a q tile takes
    static constexpr int RING = NSLOT * SLOT;
    static constexpr int PREP = NW;                       // control warps: PREP, then the decider
    static constexpr int THREADS = (NW + 2) * 32;
    static_assert(1 + QSLOTS <= NSLOT, "a residual tile (logits + q) fits the ring");
};

// A pass the stream warps run, as the decider published it.
struct __align__(16) VPass {
    int kind;     // PASS_*
    int b;        // request
    int row;      // row j of request b (ROW) or the rejected row e (RESID)
    int buf;      // result buffer
    int greedy;   // ROW: argmax instead of the sum
    int x;        // ROW: draft token whose logit is gathered (-1: none)
    float kappa;  // log2(e) / T
    float m;      // RESID: max of row e
    float invZ;   // RESID: 1 / Z_e
    int pad[3];
};

// A claimed request, prepared by the prep warp (lane j holds row j).
struct __align__(16) VReq {
    int b, n, greedy;
    float kappa;
    int x[32];     // draft tokens (j < n)
    float qx[32];  // q_j(x_j) (sampling rows j < n)
    float u[32];   // acceptance uniform of row j (Philox lane 0)
    float u2[32];  // emission uniform of row j (Philox lane 1)
};

// Shared state of the control protocol (static shared memory).
struct VCtl {
    VPass desc[VDRING];
    VReq req[VREQ];
    float lx[VBUF];            // gathered l_j(x_j) of a ROW pass
    int pub;                   // passes published
    int abort;                 // a bounded wait ran out somewhere
    int prep_done;             // no request left to claim
    int want;                  // requests the decider has asked for so far
    int given;                 // claims the prep warp has made so far
    int state[VREQ];           // REQ_*
    int ntrace;                // SV_TRACE records written by this CTA
    // the decider's own record of each request record's pass in flight
    int dkind[VREQ], dbuf[VREQ], drow[VREQ], debuf[VREQ];
    float dM[VREQ], dZ[VREQ];  // (max, Z) of the rejected row of a residual
    uint64_t done[VBUF];       // a pass's result buffer is complete (NW arrivals)
    uint64_t dbar;             // the decider's draw stage
};

__device__ __forceinline__ int vload(const int* p) { return *reinterpret_cast<const volatile int*>(p); }
// A control word as lane 0 of the calling warp reads it, for every lane (all
// 32 lanes call it): lanes that read a word another warp is changing each on
// their own may see different values, and the warp's control flow splits.
__device__ __forceinline__ int vload_w(const int* p) { return __shfl_sync(0xffffffffu, vload(p), 0); }
// A bounded wait that started at t0 has run out, by lane 0's clock (all 32
// lanes call it, so the warp leaves the wait as one).
__device__ __forceinline__ bool waited_out(uint64_t t0) {
    return __shfl_sync(0xffffffffu, int(globaltimer_ns() - t0 > VWAIT_NS), 0) != 0;
}
__device__ __forceinline__ void vstore(int* p, int v) { *reinterpret_cast<volatile int*>(p) = v; }

__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Build option SV_TRACE: each CTA records its control events (request ready,
// pass published, pass complete, request finished) with globaltimer stamps in
// the workspace's tile-partial section, which this kernel does not otherwise
// use: 256 records of 16 bytes per CTA (timing studies only; off by default).
enum { TR_READY = 1, TR_PUB = 2, TR_DONE = 3, TR_FIN = 4, TR_SSTART = 5, TR_SLAND = 6,
       TR_SARR = 7, TR_ENTRY = 11, TR_GO = 12, TR_PER_CTA = 256 };
__device__ __forceinline__ void trace(const Params& P, int* count, int kind, int b, int row) {
#ifdef SV_TRACE
    const int i = atomicAdd(count, 1);
    if (i < TR_PER_CTA)
        reinterpret_cast<uint4*>(P.part)[(size_t)blockIdx.x * TR_PER_CTA + i] =
            make_uint4(uint32_t(globaltimer_ns()), uint32_t(kind), uint32_t(b), uint32_t(row));
#else
    (void)P, (void)count, (void)kind, (void)b, (void)row;
#endif
}

}  // namespace

// Before k_verify: clear the claim counter and the status word, and write the
// claim order: requests with more drafts first (counting sort on num_draft,
// stable in b), so that the longest verifications start first.  One CTA.
__global__ void __launch_bounds__(1024) k_prep(Params P) {
    __shared__ int cnt[SPEC_MAX_K + 2];
    __shared__ int base[SPEC_MAX_K + 2];
    griddep_launch_dependents();
    const int tid = threadIdx.x;
    if (tid < SPEC_MAX_K + 2) cnt[tid] = 0;
    if (tid == 0) {
        P.hdr[HDR_VCLAIM] = 0;
        *P.status = 0;
    }
    __syncthreads();
    // bucket k holds num_draft = K - k (bad counts go to the last bucket)
    const int NB = P.K + 2;
    for (int b = tid; b < P.B; b += blockDim.x) {
        const int n = P.num_draft[b];
        const int k = (n >= 0 && n <= P.K) ? P.K - n : NB - 1;
        atomicAdd(&cnt[k], 1);
    }
    __syncthreads();
    if (tid == 0) {
        int s = 0;
        for (int k = 0; k < NB; ++k) {
            base[k] = s;
            s += cnt[k];
        }
    }
    __syncthreads();
    // stable placement: warp-sequential over b in blocks of blockDim
    for (int b0 = 0; b0 < P.B; b0 += blockDim.x) {
        const int b = b0 + tid;
        int k = -1;
        if (b < P.B) {
            const int n = P.num_draft[b];
            k = (n >= 0 && n <= P.K) ? P.K - n : NB - 1;
        }
        for (int kk = 0; kk < NB; ++kk) {
            const bool mine = (k == kk);
            // rank of this thread among the block's threads in bucket kk
            const unsigned bal = __ballot_sync(0xffffffffu, mine);
            __shared__ int wcount[32];
            const int warp = tid >> 5, lane = tid & 31;
            if (lane == 0) wcount[warp] = __popc(bal);
            __syncthreads();
            int before = 0;
            for (int w2 = 0; w2 < warp; ++w2) before += wcount[w2];
            if (mine) P.rowlist[base[kk] + before + __popc(bal & ((1u << lane) - 1u))] = b;
            __syncthreads();
            if (tid == 0) {
                int tot = 0;
                for (int w2 = 0; w2 < int(blockDim.x >> 5); ++w2) tot += wcount[w2];
                base[kk] += tot;
            }
            __syncthreads();
        }
    }
}

namespace {

// Residual mass of one staged tile (logits at st, q at stq, nel tokens) by one
// warp: lane l takes the 8-token groups k * 32 + l, sums each group's
// max(0, p - q) pairwise, then its 8 groups pairwise; the lanes by shuffles.
// resid() is the expression the level-2 scan of draw.cuh evaluates.
template <int DT>
__device__ __forceinline__ float resid_tile_mass(const uint8_t* st, const uint8_t* stq, int nel,
                                                 float m, float kappa, float invZ) {
    const int lane = threadIdx.x & 31;
    const float cm = offset_of(m, kappa);
    float gs[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int g = k * 32 + lane;
        gs[k] = 0.f;
        if (g * 8 < nel) {
            float l[8], q[8];
            smem_logits8<DT>(st, g, l);
            smem_q8(stq, g, q);
#pragma unroll
            for (int e = 0; e < 8; ++e) l[e] = resid(l[e], q[e], m, cm, kappa, invZ);
#pragma unroll
            for (int h = 4; h; h >>= 1)
#pragma unroll
                for (int e = 0; e < h; ++e) l[e] = __fadd_rn(l[e], l[e + h]);
            gs[k] = l[0];
        }
    }
#pragma unroll
    for (int h = 4; h; h >>= 1)
#pragma unroll
        for (int k = 0; k < h; ++k) gs[k] = __fadd_rn(gs[k], gs[k + h]);
    return warp_sum_f(gs[0]);
}

// Bounded wait until pass p is published (false: abort or timeout).
__device__ __forceinline__ bool wait_published(VCtl& S, int p, const Params& P) {
    if (vload_w(&S.pub) > p) return true;
    const uint64_t t0 = globaltimer_ns();
    while (vload_w(&S.pub) <= p) {
        if (vload_w(&S.abort)) return false;
        if (waited_out(t0)) {
            vstore(&S.abort, 1);
            if ((threadIdx.x & 31) == 0) atomicOr(P.status, int(SPEC_BADBIT_TIMEOUT));
            return false;
        }
        __nanosleep(64);
    }
    return true;
}

// A stream warp: runs the published passes in order.  Its producer state
// (warp-uniform; lane 0 issues the copies) walks the passes ahead of the
// consumer as far as its ring allows: a ROW tile takes one slot (slots in
// rotation), a RESID tile (logits + q) the whole ring from slot 0, issued once
// the ring is empty.  A FIFO of the issued tiles ({chunk, slot, kind}, 10 bits
// each) gives the consumer the slot of each tile in issue order.
template <int DT>
__device__ __forceinline__ void v_stream(const Params& P, VCtl& S, Partial* bufs, uint8_t* ring,
                                         uint64_t* bars, int w) {
    using CF = VCfg<DT>;
    using TL = Tile<DT>;
    constexpr int NW = CF::NW, NSLOT = CF::NSLOT, EPV = TL::EPV, VPL = TL::VPL;
    const int lane = threadIdx.x & 31;
    const int C = P.C, V = P.V;

    int ip = 0, ik = 0;      // producer: pass and tile index (chunk w + ik * NW) to issue next
    bool pend = true;        // the producer has not reached the end pass
    int head = 0, nfree = NSLOT;
    uint32_t fifo = 0, busy = 0;  // busy: slots with a copy not yet waited for
    int fn = 0;
    uint32_t phase = 0;      // bit s: parity of slot s's next completion

    auto try_issue = [&]() {
        while (pend) {
            if (ip >= vload_w(&S.pub)) break;
            __threadfence_block();
            const VPass& d = S.desc[ip % VDRING];
            const int kind = d.kind;
            if (kind == PASS_END) {
                pend = false;
                break;
            }
            const int c = w + ik * NW;
            if (c >= C) {
                ++ip;
                ik = 0;
                continue;
            }
            const bool rs = kind == PASS_RESID;
            if (rs ? nfree < NSLOT : nfree == 0) break;
            const int slot = rs ? 0 : head;
            const int nel = min(TILE, V - c * TILE);
            if (lane == 0) {
                const size_t row = (size_t)d.b * P.K1 + d.row;
                const uint32_t lb = uint32_t(nel) * CF::ESZ, qb = rs ? uint32_t(nel) * 4u : 0u;
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&bars[slot], lb + qb);
                bulk_g2s(ring + slot * CF::SLOT,
                         reinterpret_cast<const char*>(P.logits) +
                             (row * V + (size_t)c * TILE) * CF::ESZ,
                         lb, &bars[slot]);
                if (rs)
                    bulk_g2s(ring + CF::SLOT,
                             P.probs + ((size_t)d.b * P.K + d.row) * V + (size_t)c * TILE, qb,
                             &bars[slot]);
            }
            if (rs) {
                nfree = 0;
                head = 0;
            } else {
                --nfree;
                head = head + 1 == NSLOT ? 0 : head + 1;
            }
            busy |= 1u << slot;
            fifo |= uint32_t(c | (slot << 7) | (rs ? 512 : 0)) << (10 * fn);
            ++fn;
            ++ik;
        }
    };

    bool ok = true;
    for (int p = 0;; ++p) {
        if (!wait_published(S, p, P)) {
            ok = false;
            break;
        }
        __threadfence_block();
        const VPass d = S.desc[p % VDRING];
        if (d.kind == PASS_END) break;
        if (w == 0 && lane == 0) trace(P, &S.ntrace, TR_SSTART, d.b, d.kind * 100 + d.row);
        const bool rs = d.kind == PASS_RESID;
        const int ntiles = C > w ? (C - 1 - w) / NW + 1 : 0;
        Partial* out = bufs + d.buf * VCMAX;
        for (int t = 0; t < ntiles; ++t) {
            if (fn == 0) try_issue();  // then the tile is in the FIFO (its pass is published)
            const uint32_t e = fifo & 1023u;
            fifo >>= 10;
            --fn;
            const int c = int(e & 127u), slot = int((e >> 7) & 3u);
            const bool landed = mbar_wait_bounded(&bars[slot], (phase >> slot) & 1u, VWAIT_NS);
            if (!__all_sync(0xffffffffu, landed)) {
                ok = false;
                break;
            }
            phase ^= 1u << slot;
            busy &= ~(1u << slot);
            if (t == 0 && w == 0 && lane == 0) trace(P, &S.ntrace, TR_SLAND, d.b, p);
            const int nel = min(TILE, V - c * TILE);
            const uint8_t* st = ring + slot * CF::SLOT;
            if (!rs) {
                const int nvec = nel / EPV;
                const uint4* v4 = reinterpret_cast<const uint4*>(st);
                uint4 dv[VPL];
                if (nvec == VPL * 32) {  // a full tile (every tile but a row's last)
#pragma unroll
                    for (int k = 0; k < VPL; ++k) dv[k] = v4[k * 32 + lane];
                } else {
#pragma unroll
                    for (int k = 0; k < VPL; ++k) {
                        const int v = k * 32 + lane;
                        dv[k] = v < nvec ? v4[v]
                                         : make_uint4(TL::NEG_INF_WORD, TL::NEG_INF_WORD,
                                                      TL::NEG_INF_WORD, TL::NEG_INF_WORD);
                    }
                }
                const bool has_x = d.x >= 0 && d.x / TILE == c;
                float lx = 0.f;
                if (has_x && lane == 0) {
                    const int ex = d.x - c * TILE;
                    if constexpr (DT == SPEC_BF16)
                        lx = __uint_as_float(uint32_t(reinterpret_cast<const uint16_t*>(st)[ex]) << 16);
                    else
                        lx = reinterpret_cast<const float*>(st)[ex];
                }
                __syncwarp();  // every lane holds its share: the slot can be refilled
                ++nfree;
                try_issue();
                const Partial pt = tile_partial<DT>(dv, nvec, c * TILE, d.greedy != 0, d.kappa);
                if (lane == 0) {
                    out[c] = pt;
                    if (has_x) S.lx[d.buf] = lx;
                }
            } else {
                const float mass = resid_tile_mass<DT>(st, st + CF::SLOT, nel, d.m, d.kappa, d.invZ);
                __syncwarp();
                nfree = NSLOT;
                head = 0;
                if (lane == 0) {
                    Partial pt;
                    pt.m = 0.f;
                    pt.amax = -1;
                    pt.z = double(mass);
                    out[c] = pt;
                }
            }
        }
        if (!ok) break;
        try_issue();  // the producer leaves pass p before the pass can complete
        __syncwarp();
        if (lane == 0) mbar_arrive_cta(&S.done[d.buf]);
        if (w == 0 && lane == 0) trace(P, &S.ntrace, TR_SARR, d.b, p);
    }
    if (!ok) {
        if (lane == 0) atomicOr(P.status, int(SPEC_BADBIT_TIMEOUT));
        vstore(&S.abort, 1);
        // let the copies still in flight land before the shared memory is released
        for (int sl = 0; sl < NSLOT; ++sl)
            if (busy & (1u << sl)) mbar_wait_bounded(&bars[sl], (phase >> sl) & 1u, 100000000ull);
    }
}

}  // namespace

namespace {

__device__ __forceinline__ void v_timeout(const Params& P, VCtl& S) {
    vstore(&S.abort, 1);
    if ((threadIdx.x & 31) == 0) atomicOr(P.status, int(SPEC_BADBIT_TIMEOUT));
}

// The prep warp: one claim per request the decider asks for.  A request that
// fails validation (num_draft, temperature, draft ids, missing q) gets its
// -1 outputs here and never reaches the decider.  Lane j holds row j.
__device__ __forceinline__ void v_prep(const Params& P, VCtl& S) {
    const int lane = threadIdx.x & 31;
    const float NaN = __int_as_float(0x7fc00000);
    int given = 0;
    for (;;) {
        uint64_t t0 = globaltimer_ns();
        bool go = true;
        for (;;) {  // lane 0 reads the shared flags: the warp takes one decision
            int st = 0;  // 1 asked, 2 abort
            if (lane == 0) st = vload(&S.want) > given ? 1 : vload(&S.abort) ? 2 : 0;
            st = __shfl_sync(0xffffffffu, st, 0);
            if (st == 1) break;
            if (st == 2 || waited_out(t0)) {
                if (st != 2) v_timeout(P, S);
                go = false;
                break;
            }
            __nanosleep(64);
        }
        if (!go) break;
        int slot = -1;
        t0 = globaltimer_ns();
        while (slot < 0 && go) {  // the decider asks only while a record is free
            int st = -1;
            if (lane == 0) {
                for (int i = VREQ - 1; i >= 0; --i)
                    if (vload(&S.state[i]) == REQ_EMPTY) st = i;
                if (st < 0 && vload(&S.abort)) st = -2;
            }
            st = __shfl_sync(0xffffffffu, st, 0);
            if (st >= 0) slot = st;
            else if (st == -2) go = false;
            else if (waited_out(t0)) {
                v_timeout(P, S);
                go = false;
            }
        }
        if (!go) break;
        int k = 0;
        if (lane == 0) k = atomicAdd(P.hdr + HDR_VCLAIM, 1);
        k = __shfl_sync(0xffffffffu, k, 0);
        if (k >= P.B) {
            if (lane == 0) {
                vstore(&S.prep_done, 1);
                __threadfence_block();
                vstore(&S.given, given + 1);
            }
            break;
        }
        const int b = P.rowlist[k];  // k_prep's claim order
        const int n = P.num_draft[b];
        const float T = P.temp[b];
        int flags = 0;
        if (n < 0 || n > P.K) flags |= SPEC_BADBIT_NUM_DRAFT;
        if (!(T >= 0.f) || T > FLT_MAX) flags |= SPEC_BADBIT_TEMPERATURE;
        const bool greedy = (T == 0.f);
        if (!flags && !greedy && n > 0 && P.probs == nullptr) flags |= SPEC_BADBIT_NO_PROBS;
        const int nn = flags ? 0 : n;
        int x = -1;
        if (lane < nn) x = P.ids[(size_t)b * P.K + lane];
        if (__any_sync(0xffffffffu, lane < nn && (x < 0 || x >= P.V))) flags |= SPEC_BADBIT_DRAFT_ID;
        float qx = 0.f, u = 0.f, u2 = 0.f;
        if (!flags && !greedy) {
            if (lane < n) qx = __ldg(P.probs + ((size_t)b * P.K + lane) * P.V + x);
            if (lane <= n) {
                const uint4 rb = row_block(P, b, lane);
                u = uniform01(rb.x);
                u2 = uniform01(rb.y);
            }
        }
        if (P.dbg_rows && lane < P.K1) {  // untested until the decider tests the row
            float* d = P.dbg_rows + ((size_t)b * P.K1 + lane) * 4;
            d[0] = d[1] = d[2] = NaN;
            d[3] = -1.f;
        }
        if (flags) {
            if (lane < P.K1) P.out_ids[(size_t)b * P.K1 + lane] = -1;
            if (lane == 0) {
                P.out_nacc[b] = -1;
                atomicOr(P.status, flags);
                if (P.dbg_req) {
                    float* d = P.dbg_req + (size_t)b * 4;
                    d[0] = float(MODE_BAD);
                    d[1] = d[2] = d[3] = NaN;
                }
                vstore(&S.given, given + 1);  // the decider asks again
            }
            ++given;
            __syncwarp();
            continue;
        }
        VReq& R = S.req[slot];
        R.x[lane] = x;
        R.qx[lane] = qx;
        R.u[lane] = u;
        R.u2[lane] = u2;
        if (lane == 0) {
            R.b = b;
            R.n = n;
            R.greedy = greedy ? 1 : 0;
            R.kappa = greedy ? 0.f : kappa_of(T);
        }
        __syncwarp();
        __threadfence_block();
        if (lane == 0) {
            trace(P, &S.ntrace, TR_READY, b, n);
            vstore(&S.state[slot], REQ_READY);
            __threadfence_block();
            vstore(&S.given, given + 1);
        }
        ++given;
        __syncwarp();
    }
}

}  // namespace

namespace {

// The decider warp (all lanes run the same control flow; lane 0 writes the
// shared control state).  Each request record has at most one pass in flight
// and passes complete in the order they were published (every stream warp
// runs them in order), so the passes in flight form a FIFO of records.
template <int DT>
__device__ __forceinline__ void v_decide(const Params& P, VCtl& S, const Partial* bufs,
                                         uint8_t* dst) {
    using ST = Stage<DT>;
    const int lane = threadIdx.x & 31;
    const int C = P.C, K1 = P.K1;
    const float NaN = __int_as_float(0x7fc00000);
    int pub = 0, want = 0;
    uint32_t bph = 0;   // bit i: parity of result buffer i's next completion
    uint32_t dph = 0;   // parity of the draw stage's barrier
    bool dbusy = false; // a draw-stage copy has not been waited for
    int f0 = -1, f1 = -1, fn = 0;
    bool ok = true;

    auto publish = [&](int kind, int s, int r, int buf, float M, float Z) {
        if (lane == 0) {
            trace(P, &S.ntrace, TR_PUB, kind == PASS_END ? -1 : S.req[s].b, kind * 100 + r);
            VPass& d = S.desc[pub % VDRING];
            d.kind = kind;
            if (kind != PASS_END) {
                const VReq& R = S.req[s];
                d.b = R.b;
                d.row = r;
                d.buf = buf;
                d.greedy = R.greedy;
                d.x = (kind == PASS_ROW && !R.greedy && r < R.n) ? R.x[r] : -1;
                d.kappa = R.kappa;
                d.m = M;
                d.invZ = float(1.0 / double(Z));
                S.dkind[s] = kind;
                S.dbuf[s] = buf;
                S.drow[s] = r;
            }
            __threadfence_block();
            vstore(&S.pub, pub + 1);
        }
        __syncwarp();
        ++pub;
        if (kind != PASS_END) {
            if (fn == 0) f0 = s;
            else f1 = s;
            ++fn;
        }
    };
    // ask the prep warp for the next request, unless a claim is pending, a
    // request is already waiting, or every record is taken
    auto ask = [&]() {
        if (vload_w(&S.given) != want || vload_w(&S.prep_done)) return;
        int taken = 0;
        bool ready = false;
        for (int i = 0; i < VREQ; ++i) {
            const int st = vload_w(&S.state[i]);
            taken += st != REQ_EMPTY;
            ready |= st == REQ_READY;
        }
        if (ready || taken >= VREQ) return;
        ++want;
        if (lane == 0) vstore(&S.want, want);
        __syncwarp();
    };
    // start every prepared request: its row 0 (the request's last row when it
    // has no drafts, and then the next request is asked for at once)
    auto activate = [&]() {
        for (int s = 0; s < VREQ; ++s) {
            if (vload_w(&S.state[s]) != REQ_READY) continue;
            __threadfence_block();
            if (lane == 0) vstore(&S.state[s], REQ_ACTIVE);
            __syncwarp();
            publish(PASS_ROW, s, 0, 2 * s, 0.f, 0.f);
            if (S.req[s].n == 0) ask();
        }
    };
    auto finish = [&](int s) {
        if (lane == 0) trace(P, &S.ntrace, TR_FIN, S.req[s].b, 0);
        __syncwarp();
        __threadfence_block();
        if (lane == 0) vstore(&S.state[s], REQ_EMPTY);
        __syncwarp();
        ask();
    };
    auto fail = [&](int s, int flags) {
        const int b = S.req[s].b;
        if (lane < K1) P.out_ids[(size_t)b * K1 + lane] = -1;
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
    // the emitted token at position a, the -1 tail, a_b and the request record
    auto emit = [&](int s, int a, int tok, int mode, double mass) {
        const VReq& R = S.req[s];
        const int b = R.b;
        if (lane == a) P.out_ids[(size_t)b * K1 + a] = tok;
        else if (lane > a && lane < K1) P.out_ids[(size_t)b * K1 + lane] = -1;
        if (lane == 0) {
            P.out_nacc[b] = a;
            if (P.dbg_req) {
                float* d = P.dbg_req + (size_t)b * 4;
                if (R.greedy) {
                    d[0] = float(MODE_GREEDY);
                    d[1] = float(a);
                    d[2] = d[3] = NaN;
                } else {
                    d[0] = float(mode);
                    d[1] = float(a);
                    d[2] = float(mass);
                    d[3] = R.u2[a];
                }
            }
        }
    };
    // copy a chunk (logits, and q when qb > 0) into the draw stage
    auto stage = [&](const void* l, uint32_t lb, const void* q, uint32_t qb) -> bool {
        if (lane == 0) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&S.dbar, lb + qb);
            bulk_g2s(dst, l, lb, &S.dbar);
            if (qb) bulk_g2s(dst + ST::LB, q, qb, &S.dbar);
        }
        dbusy = true;
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&S.dbar, dph, VWAIT_NS))) {
            v_timeout(P, S);
            return false;
        }
        dph ^= 1u;
        dbusy = false;
        return true;
    };
    // a draw from p of row `row` of request b, given the row's tile partials
    // and its (max, kappa): level 1 over the rebased tile sums, level 2 over
    // the chosen tile (copied again, from L2)
    auto draw_p = [&](const Partial* part, int b, int row, float M, float kappa, float u2,
                      double& total) -> int {
        const Pick pk = pick_chunk(C, u2, [&](int c) -> double {
            const Partial q = part[c];
            if (q.m == -INFINITY || q.z == 0.0) return 0.0;
            return q.z * double(rebase_factor(q.m, M, kappa));
        });
        total = pk.total;
        if (pk.chunk < 0) return 0;  // no mass at all (not for a row with a finite logit)
        const Partial pc = part[pk.chunk];
        const double f_c = double(rebase_factor(pc.m, M, kappa));
        const double t = (double(u2) * pk.total - pk.before) * pow2_recip(f_c);
        const float cc = offset_of(pc.m, kappa);
        const int c0 = pk.chunk * TILE, nel = min(TILE, P.V - c0);
        const char* src = reinterpret_cast<const char*>(P.logits) +
                          (((size_t)b * K1 + row) * P.V + c0) * ST::ESZ;
        if (!stage(src, uint32_t(nel) * ST::ESZ, nullptr, 0)) return 0;
        const int x = level2(c0, nel, t, [&](int g, float (&w)[8]) {
            float l[8];
            smem_logits8<DT>(dst, g, l);
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = ex2_approx(weight_arg(l[k], pc.m, cc, kappa));
        });
        __syncwarp();
        return x;
    };

    auto on_row = [&](int s) {
        const VReq& R = S.req[s];
        const int j = S.drow[s], buf = S.dbuf[s];
        const int n = R.n, b = R.b;
        const bool greedy = R.greedy != 0;
        const float kappa = R.kappa;
        const Partial* pp = bufs + buf * VCMAX;
        Partial q[MERGE_NPL];
#pragma unroll
        for (int i = 0; i < MERGE_NPL; ++i) {
            const int c = lane + 32 * i;
            if (c < C) {
                q[i] = pp[c];
            } else {
                q[i].m = -INFINITY;
                q[i].amax = INT_MAX;
                q[i].z = 0.0;
            }
        }
        float M, Z;
        int A;
        merge_loaded(q, greedy, kappa, M, Z, A);
        if (!greedy && M == -INFINITY) {  // a sampling row with no finite logit
            fail(s, SPEC_BADBIT_EMPTY_ROW);
            finish(s);
            return;
        }
        if (j < n) {  // the test of draft j
            const int x = R.x[j];
            bool acc;
            float pj = NaN, u = NaN;
            if (greedy) {
                acc = (x == A);
            } else {
                const float lx = S.lx[buf], qx = R.qx[j];
                pj = __fdiv_rn(exp2f(weight_arg(lx, M, offset_of(M, kappa), kappa)), Z);
                u = R.u[j];
                // u <= p / q  <=>  u q <= p (q > 0), exact as a product in float64
                acc = (pj > 0.f) && (qx == 0.f || double(u) * double(qx) <= double(pj));
            }
            if (P.dbg_rows && lane == 0) {
                float* d = P.dbg_rows + ((size_t)b * K1 + j) * 4;
                d[0] = greedy ? NaN : pj;
                d[1] = greedy ? NaN : u;
                d[2] = greedy ? NaN : Z;
                d[3] = acc ? 1.f : 0.f;
            }
            if (acc) {
                if (lane == 0) P.out_ids[(size_t)b * K1 + j] = x;
                publish(PASS_ROW, s, j + 1, 2 * s + ((j + 1) & 1), 0.f, 0.f);
                if (j + 1 == n) ask();  // the request's last row is on its way
                return;
            }
            if (greedy) {  // the target's argmax replaces the first mismatch
                emit(s, j, A, MODE_GREEDY, 0.0);
                finish(s);
                return;
            }
            // rejected: the residual max(0, p_j - q_j) over row j, still in L2
            if (lane == 0) {
                S.dM[s] = M;
                S.dZ[s] = Z;
                S.debuf[s] = buf;
            }
            __syncwarp();
            publish(PASS_RESID, s, j, 2 * s + ((j + 1) & 1), M, Z);
            ask();
            return;
        }
        // every draft kept: the bonus token from row n
        if (greedy) {
            emit(s, n, A, MODE_GREEDY, 0.0);
        } else {
            double total = 0.0;
            const int tok = draw_p(pp, b, n, M, kappa, R.u2[n], total);
            if (vload_w(&S.abort)) return;
            emit(s, n, tok, MODE_BONUS, total);
        }
        finish(s);
    };

    auto on_resid = [&](int s) {
        const VReq& R = S.req[s];
        const int e = S.drow[s], b = R.b;
        const float kappa = R.kappa, u2 = R.u2[e];
        const float M = S.dM[s], Z = S.dZ[s];
        const Partial* mp = bufs + S.dbuf[s] * VCMAX;
        double pre[PICK_NB];
        load_masses(C, [&](int c) -> double { return mp[c].z; }, pre);
        const Pick pk = pick_loaded(u2, pre);
        if (pk.chunk < 0) {  // a residual without mass: draw from p of row e instead
            double total = 0.0;
            const int tok = draw_p(bufs + S.debuf[s] * VCMAX, b, e, M, kappa, u2, total);
            if (vload_w(&S.abort)) return;
            emit(s, e, tok, MODE_FALLBACK, total);
            finish(s);
            return;
        }
        const double t = double(u2) * pk.total - pk.before;
        const float invZ = float(1.0 / double(Z));
        const float cm = offset_of(M, kappa);
        const int c0 = pk.chunk * TILE, nel = min(TILE, P.V - c0);
        const char* l = reinterpret_cast<const char*>(P.logits) +
                        (((size_t)b * K1 + e) * P.V + c0) * ST::ESZ;
        const float* q = P.probs + ((size_t)b * P.K + e) * P.V + c0;
        if (!stage(l, uint32_t(nel) * ST::ESZ, q, uint32_t(nel) * 4u)) return;
        const int x = level2(c0, nel, t, [&](int g, float (&w)[8]) {
            float lv[8], qv[8];
            smem_logits8<DT>(dst, g, lv);
            smem_q8(dst + ST::LB, g, qv);
#pragma unroll
            for (int k = 0; k < 8; ++k) w[k] = resid(lv[k], qv[k], M, cm, kappa, invZ);
        });
        __syncwarp();
        emit(s, e, x, MODE_RESIDUAL, pk.total);
        finish(s);
    };

    ask();  // the first request
    uint64_t idle0 = globaltimer_ns();
    for (;;) {
        activate();
        if (fn == 0) {
            bool all_empty = true;
            for (int i = 0; i < VREQ; ++i) all_empty &= vload_w(&S.state[i]) == REQ_EMPTY;
            if (all_empty && vload_w(&S.prep_done)) {
                publish(PASS_END, 0, 0, 0, 0.f, 0.f);
                break;
            }
            ask();
            if (vload_w(&S.abort)) {
                ok = false;
                break;
            }
            if (waited_out(idle0)) {
                v_timeout(P, S);
                ok = false;
                break;
            }
            __nanosleep(32);
            continue;
        }
        const int s = f0;
        const int buf = S.dbuf[s];
        const uint32_t par = (bph >> buf) & 1u;
        const uint64_t t0 = globaltimer_ns();
        bool got = true;
        while (!__all_sync(0xffffffffu, mbar_try_wait(&S.done[buf], par))) {
            activate();
            if (vload_w(&S.abort)) {
                got = false;
                break;
            }
            if (waited_out(t0)) {
                v_timeout(P, S);
                got = false;
                break;
            }
        }
        if (!got) {
            ok = false;
            break;
        }
        bph ^= 1u << buf;
        if (lane == 0) trace(P, &S.ntrace, TR_DONE, S.req[s].b, S.dkind[s] * 100 + S.drow[s]);
        f0 = f1;
        --fn;
        if (S.dkind[s] == PASS_ROW) on_row(s);
        else on_resid(s);
        if (vload_w(&S.abort)) {
            ok = false;
            break;
        }
        idle0 = globaltimer_ns();
    }
    if (!ok && dbusy)  // let a draw copy still in flight land
        mbar_wait_bounded(&S.dbar, dph, 100000000ull);
}

template <int DT>
__device__ __forceinline__ void verify_body(const Params& P) {
    using CF = VCfg<DT>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ VCtl S;
    __shared__ __align__(8) uint64_t bars[CF::NW][CF::NSLOT];
    uint8_t* dstage = smem + size_t(CF::NW) * CF::RING;
    Partial* bufs = reinterpret_cast<Partial*>(dstage + Stage<DT>::BYTES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        S.pub = 0;
        S.abort = 0;
        S.prep_done = 0;
        S.want = 0;
        S.given = 0;
        S.ntrace = 0;
        for (int i = 0; i < VREQ; ++i) S.state[i] = REQ_EMPTY;
        for (int i = 0; i < VBUF; ++i) mbar_init(&S.done[i], CF::NW);
        mbar_init(&S.dbar, 1);
        fence_mbarrier_init();
    }
    if (warp < CF::NW && lane == 0) {
        for (int k = 0; k < CF::NSLOT; ++k) mbar_init(&bars[warp][k], 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) trace(P, &S.ntrace, TR_ENTRY, 0, 0);
    griddep_wait();  // k_prep's claim order and cleared counter
    if (threadIdx.x == 0) trace(P, &S.ntrace, TR_GO, 0, 0);
    if (warp < CF::NW)
        v_stream<DT>(P, S, bufs, smem + size_t(warp) * CF::RING, bars[warp], warp);
    else if (warp == CF::PREP)
        v_prep(P, S);
    else
        v_decide<DT>(P, S, bufs, dstage);
}

}  // namespace

size_t verify_smem(int dtype) {
    return dtype == SPEC_BF16
               ? size_t(VCfg<SPEC_BF16>::NW) * VCfg<SPEC_BF16>::RING + Stage<SPEC_BF16>::BYTES +
                     size_t(VBUF) * VCMAX * sizeof(Partial)
               : size_t(VCfg<SPEC_F32>::NW) * VCfg<SPEC_F32>::RING + Stage<SPEC_F32>::BYTES +
                     size_t(VBUF) * VCMAX * sizeof(Partial);
}
int verify_threads(int dtype) {
    return dtype == SPEC_BF16 ? VCfg<SPEC_BF16>::THREADS : VCfg<SPEC_F32>::THREADS;
}

__global__ void __launch_bounds__(VCfg<SPEC_BF16>::THREADS, 1) k_verify_bf16(Params P) {
    verify_body<SPEC_BF16>(P);
}
__global__ void __launch_bounds__(VCfg<SPEC_F32>::THREADS, 1) k_verify_f32(Params P) {
    verify_body<SPEC_F32>(P);
}

}  // namespace sv
