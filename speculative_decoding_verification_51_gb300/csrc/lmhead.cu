// lmhead.cu -- the target's logits produced on the tensor cores: an LM-head
// GEMM, logits[r, v] = sum_h hidden[r, h] * W[v, h], for the rows the verifier
// reads, with bf16 operands and float32 accumulation.
//
// The pages score the drafts with one target forward that yields p_1 ..
// p_{gamma+1} ("投机采样", 第二步; "深入推测解码" 保证原始分布 step 2); the
// logits of that forward are the last layer's hidden states times the
// vocabulary projection.  This file makes that projection on sm_103a:
//   - operands are staged by TMA (cp.async.bulk.tensor, 128-byte swizzle,
//     4-stage ring, one mbarrier per stage and direction);
//   - one thread issues tcgen05.mma (kind::f16, M = 128, N = 256, K = 16,
//     both operands K-major) into a TMEM accumulator; tcgen05.commit frees a
//     stage when the MMAs reading it are done;
//   - two accumulators of 256 columns alternate, so the epilogue (4 warps,
//     tcgen05.ld, one row per thread) drains one while the next is computed.
// A CTA computes a 128-row x 2048-column block: 8 sub-tiles of 256 columns,
// one TMA box of A (128 x 64) and B (256 x 64) per K step of 64.
//
// The fused form (spec_verify_lmhead) reads the rows k_plan listed, writes
// each row's logits at its slot, and in the same epilogue takes the
// statistics k_row_stats would take from those logits: per (row, 2048-token
// chunk) the maximum and, for sampling rows, the sum of 2^(l*kappa - c)
// against c = offset_of(chunk max, kappa) (kept online over the chunk's 32-column
// pieces, rescaled when the maximum grows), or for greedy rows the lowest
// index of the maximum; l(x_j) and q(x_j) for the draft token.  All of it
// is computed from the bf16-rounded logits that are stored, so the later
// residual and bonus draws see the same values.  k_accept_all then runs
// every request's acceptance (accept_request), one warp per request: run by
// the epilogue warps themselves, a warp that completed several requests at
// once ran their acceptances one after another at the end of the GEMM.
//
// Every wait is bounded: a CTA that times out sets SPEC_BADBIT_TIMEOUT, lets
// its copies and MMAs in flight finish (again bounded), frees its TMEM and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <climits>
#include <mutex>

#include "accept.cuh"
#include "common.cuh"

namespace sv {

namespace {

constexpr int LM_BM = 128, LM_BN = 256, LM_BK = 64, LM_STAGES = 4;
constexpr int LM_A_BYTES = LM_BM * LM_BK * 2;             // 16 KB
constexpr int LM_B_BYTES = LM_BN * LM_BK * 2;             // 32 KB
constexpr int LM_STAGE_BYTES = LM_A_BYTES + LM_B_BYTES;   // 48 KB
constexpr int LM_THREADS = 192;  // warp 0: TMA, warp 1: MMA + TMEM, warps 2..5: epilogue
constexpr int LM_TMEM_COLS = 2 * LM_BN;
constexpr uint64_t LM_WAIT_NS = 200000000ull;  // 0.2 s per wait
constexpr size_t LM_SMEM = 1024 + size_t(LM_STAGES) * LM_STAGE_BYTES;

// kind::f16 instruction descriptor: D f32, A and B bf16, both K-major, N, M.
__host__ __device__ constexpr uint32_t lm_idesc() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(LM_BN >> 3) << 17) |
           (uint32_t(LM_BM >> 4) << 24);
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with the 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = uint64_t((saddr >> 4) & 0x3FFFu);
    d |= uint64_t(1) << 16;             // leading byte offset (unused by this swizzle)
    d |= uint64_t(1024 >> 4) << 32;     // stride byte offset: next 8-row group
    d |= uint64_t(1) << 46;             // descriptor version
    d |= uint64_t(2) << 61;             // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// 32 consecutive accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Two floats -> packed bf16x2 (round to nearest even): lo in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

struct LmArgs {
    int rows;             // rows of A (and of the output)
    int H, V;
    uint16_t* out;        // [rows, V] bf16 logits
    int32_t* status;      // device status word
};

}  // namespace

template <bool FUSED>
__global__ void __launch_bounds__(LM_THREADS, 1)
    k_lmhead(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             LmArgs L, Params P) {
    extern __shared__ uint8_t lm_smem_raw[];
    __shared__ __align__(8) uint64_t full[LM_STAGES], empty[LM_STAGES], accf[2], acce[2], fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the row tiles of one 2048-column block run side by side, so its slice
    // of the LM head is read from HBM once and then served from L2
    const int mt = blockIdx.x, chunk = blockIdx.y;
    const int row0 = mt * LM_BM;
    const int rows = FUSED ? P.hdr[HDR_ROWS] : L.rows;  // fused: the rows k_plan listed
    if (row0 >= rows) return;  // a row tile past the list (uniform over the CTA)
    const int col0 = chunk * TILE;
    const int ncols = min(TILE, L.V - col0);
    const int nsub = (ncols + LM_BN - 1) / LM_BN;
    const int nk = L.H / LM_BK;
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(lm_smem_raw) + 1023) & ~uintptr_t(1023));

    if (threadIdx.x == 0) {
        for (int s = 0; s < LM_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);  // released by this CTA's MMAs
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&accf[a], 1);
            mbar_init(&acce[a], 4);  // one arrival per epilogue warp
        }
        mbar_init(&fin, 1);
        abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {  // the whole warp allocates the two accumulators
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&tmem_base)),
                     "r"(LM_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    volatile int* abort_v = &abort_flag;

    if (warp == 0) {
        // ---- TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            for (int n = 0; n < nsub && !*abort_v; ++n) {
                for (int k = 0; k < nk; ++k) {
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u, LM_WAIT_NS)) {
                        *abort_v = 1;
                        break;
                    }
                    uint8_t* a = smem + size_t(s) * LM_STAGE_BYTES;
                    // the A box of this row tile and the B box of this sub-tile
                    mbar_arrive_expect_tx(&full[s], uint32_t(LM_STAGE_BYTES));
                    tma_load_2d(a, &tmA, k * LM_BK, row0, &full[s]);
                    tma_load_2d(a + LM_A_BYTES, &tmB, k * LM_BK, col0 + n * LM_BN, &full[s]);
                    if (++s == LM_STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // every stage released (so every copy has landed and no arrival is
            // still on its way) before the CTA may leave
            for (int k = 0; k < LM_STAGES; ++k) {
                mbar_wait_bounded(&empty[s], ph ^ 1u, LM_WAIT_NS);
                if (++s == LM_STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = lm_idesc();
            int s = 0;
            uint32_t ph = 0;
            bool issued_any = false;
            for (int n = 0; n < nsub && !*abort_v; ++n) {
                const int acc = n & 1;
                if (!mbar_wait_bounded(&acce[acc], (uint32_t(n >> 1) & 1u) ^ 1u, LM_WAIT_NS)) {
                    *abort_v = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tbase + uint32_t(acc * LM_BN);
                for (int k = 0; k < nk; ++k) {
                    if (!mbar_wait_bounded(&full[s], ph, LM_WAIT_NS)) {
                        *abort_v = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = smem_u32(smem + size_t(s) * LM_STAGE_BYTES);
                    const uint32_t b = a + LM_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < LM_BK / 16; ++kk)
                        tc_mma(d, sw128_desc(a + kk * 32), sw128_desc(b + kk * 32), idesc,
                               (k > 0 || kk > 0) ? 1u : 0u);
                    issued_any = true;
                    // the stage is free once these MMAs are done
                    tc_commit(&empty[s]);
                    if (++s == LM_STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (*abort_v) break;
                tc_commit(&accf[acc]);  // the sub-tile's accumulator is complete
            }
            if (issued_any) {  // every MMA of this CTA is done before TMEM is freed
                tc_commit(&fin);
                mbar_wait_bounded(&fin, 0, LM_WAIT_NS);
            }
        }
    } else {
        // ---- epilogue: TMEM -> registers -> bf16 logits, one row per thread
        const int q = warp & 3;  // the TMEM lane quarter this warp may read
        const int r = row0 + q * 32 + lane;
        const bool valid = r < rows;
        // fused: this row's slot, request and draft token
        int slot = r, b = -1, n = 0, j = 0, x = -1;
        bool greedy = true;
        float kappa = 0.f, qx = 0.f;
        if (FUSED && valid) {
            slot = P.rowlist[r];
            b = slot / P.K1;
            j = slot - b * P.K1;
            n = P.num_draft[b];
            const float T = P.temp[b];
            greedy = (T == 0.f);
            kappa = greedy ? 0.f : kappa_of(T);
            if (!greedy && j < n) {
                const int xx = P.ids[(size_t)b * P.K + j];
                if (xx >= 0 && xx < P.V && xx / TILE == chunk) x = xx;  // only this chunk's
            }
            if (x >= 0 && P.rule == RULE_LOSSLESS)
                qx = __ldg(P.probs + ((size_t)b * P.K + j) * P.V + x);
        }
        float m_run = -INFINITY, z_run = 0.f, c_run = -INFINITY, lx = 0.f;
        int amax = INT_MAX;
        bool ok = true;
        for (int nn = 0; nn < nsub; ++nn) {
            const int acc = nn & 1;
            const bool got = mbar_wait_bounded(&accf[acc], uint32_t(nn >> 1) & 1u, LM_WAIT_NS);
            if (__any_sync(0xffffffffu, !got || *abort_v)) {
                *abort_v = 1;
                ok = false;
                break;
            }
            tc_fence_after();
            const int cbase = col0 + nn * LM_BN;
#pragma unroll 1
            for (int p = 0; p < LM_BN / 32; ++p) {
                uint32_t v[32];
                tc_ld32(tbase + (uint32_t(q * 32) << 16) + uint32_t(acc * LM_BN + p * 32), v);
                const int c = cbase + p * 32;
                if (!valid || c >= L.V) continue;
                uint32_t w[16];
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    w[k] = pack_bf16x2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
                uint4* dst = reinterpret_cast<uint4*>(L.out + (size_t)slot * L.V + c);
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    if (c + g * 8 < L.V)  // V is a multiple of 8
                        dst[g] = make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
                if constexpr (FUSED) {
                    // statistics of the stored (bf16) values of this piece
                    float f[32];
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        f[2 * k] = bf16_lo(w[k]);
                        f[2 * k + 1] = bf16_hi(w[k]);
                    }
                    const int lim = min(32, L.V - c);
                    float pm = -INFINITY;
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        if (k < lim) pm = fmaxf(pm, f[k]);
                    if (greedy) {
                        if (pm > m_run) {  // the first index of the new maximum
                            int kf = 31;
#pragma unroll
                            for (int k = 31; k >= 0; --k)
                                if (k < lim && f[k] == pm) kf = k;
                            m_run = pm;
                            amax = c + kf;
                        }
                    } else {
                        if (pm > m_run) {  // rebase the running sum onto the new offset
                            if (z_run != 0.f)
                                z_run = __fmul_rn(z_run, rebase_factor(m_run, pm, kappa));
                            m_run = pm;
                            c_run = offset_of(pm, kappa);
                        }
                        float zs = 0.f;
                        if (offset_ok(c_run)) {
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                if (k < lim) zs = __fadd_rn(zs, ex2_approx(fmaf(f[k], kappa, -c_run)));
                        } else {  // offset too large (very small T): (l - max) * kappa
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                if (k < lim)
                                    zs = __fadd_rn(zs, ex2_approx(__fmul_rn(__fsub_rn(f[k], m_run), kappa)));
                        }
                        z_run = __fadd_rn(z_run, zs);
                    }
                    if (x >= c && x < c + 32) {
                        const int e = x - c;
#pragma unroll
                        for (int k = 0; k < 32; ++k)
                            if (k == e) lx = f[k];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acce[acc]);
        }
        if constexpr (FUSED) {
            if (ok) {
                if (valid) {
                    Partial o;
                    o.m = m_run;
                    o.amax = greedy ? amax : -1;
                    o.z = greedy ? 0.0 : double(z_run);
                    P.part[(size_t)slot * P.C + chunk] = o;
                    if (x >= 0) P.gath[slot] = make_float2(lx, qx);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                     "r"(LM_TMEM_COLS)
                     : "memory");
    if (threadIdx.x == 0 && *abort_v) atomicOr(L.status, int(SPEC_BADBIT_TIMEOUT));
}

// The listed rows' hidden states, in list order (one warp per row, 16-byte
// copies); rows past the list are left as they are.
__global__ void __launch_bounds__(256) k_gather_rows(Params P, LmHeadIn in) {
    const int lane = threadIdx.x & 31;
    const int R = P.hdr[HDR_ROWS];
    const int nvec = in.H / 8;
    for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < R; r += gridDim.x * 8) {
        const int slot = P.rowlist[r];
        const uint4* src = reinterpret_cast<const uint4*>(in.hidden) + (size_t)slot * nvec;
        uint4* dst = reinterpret_cast<uint4*>(in.hid_c) + (size_t)r * nvec;
        for (int i = lane; i < nvec; i += 32) dst[i] = __ldg(src + i);
    }
}

}  // namespace sv

using namespace sv;

namespace {

std::mutex g_lm_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

spec_status encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
    std::lock_guard<std::mutex> lk(g_lm_mu);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return SPEC_ERR_CUDA;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return SPEC_OK;
}

// K-major bf16 matrix [rows, H] tiled in (64 x box_rows) boxes, 128-byte swizzle.
spec_status make_map(CUtensorMap* map, const void* base, int rows, int H, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    if (encoder(&enc) != SPEC_OK) return SPEC_ERR_CUDA;
    const cuuint64_t dims[2] = {cuuint64_t(H), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(H) * 2};
    const cuuint32_t box[2] = {cuuint32_t(LM_BK), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                           strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SPEC_OK : SPEC_ERR_INVALID_ARG;
}

// Row tiles of `rows`.
int row_tiles(int rows) { return (rows + LM_BM - 1) / LM_BM; }

template <bool FUSED>
cudaError_t launch_lm(dim3 grid, cudaStream_t st, const CUtensorMap& ma, const CUtensorMap& mb,
                      const LmArgs& L, const Params& P) {
    k_lmhead<FUSED><<<grid, LM_THREADS, LM_SMEM, st>>>(ma, mb, L, P);
    return cudaGetLastError();
}

// Per-device kernel attributes (shared memory above 48 KB), set once.
spec_status lm_prepare() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SPEC_ERR_CUDA;
    static bool done[64] = {};
    std::lock_guard<std::mutex> lk(g_lm_mu);
    if (!done[dev]) {
        if (cudaFuncSetAttribute(k_lmhead<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(LM_SMEM)) != cudaSuccess ||
            cudaFuncSetAttribute(k_lmhead<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(LM_SMEM)) != cudaSuccess)
            return SPEC_ERR_CUDA;
        done[dev] = true;
    }
    return SPEC_OK;
}

}  // namespace

namespace sv {

// Gather the listed rows' hidden states, then the fused projection + row
// statistics + acceptance over them (after k_plan, before k_sample).
spec_status launch_lmhead_fused(const Params& P, const LmHeadIn& in, cudaStream_t st) {
    const int maxrows = P.B * P.K1;
    CUtensorMap ma, mb;
    spec_status r = make_map(&ma, in.hid_c, maxrows, in.H, LM_BM);
    if (r != SPEC_OK) return r;
    r = make_map(&mb, in.lm_head, P.V, in.H, LM_BN);
    if (r != SPEC_OK) return r;
    if (lm_prepare() != SPEC_OK) return SPEC_ERR_CUDA;
    const int gblocks = min((maxrows + 7) / 8, 4096);
    k_gather_rows<<<gblocks, 256, 0, st>>>(P, in);
    LmArgs L;
    L.rows = maxrows;
    L.H = in.H;
    L.V = P.V;
    L.out = static_cast<uint16_t*>(const_cast<void*>(P.logits));
    L.status = P.status;
    const dim3 grid(unsigned(row_tiles(maxrows)), unsigned(P.C));
    if (launch_lm<true>(grid, st, ma, mb, L, P) != cudaSuccess) return SPEC_ERR_CUDA;
    k_accept_all<<<P.B, ACCEPT_WARPS * 32, 0, st>>>(P);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace sv

extern "C" {

spec_status spec_lmhead_logits(const void* hidden, const void* lm_head, int rows, int H, int V,
                               void* logits_out, int32_t* dev_status, spec_stream_t stream) {
    if (rows < 0 || H <= 0 || V < 8 || rows > (1 << 24) || V > (1 << 24) || H > (1 << 16))
        return SPEC_ERR_INVALID_ARG;
    if (H % LM_BK != 0 || V % 8 != 0) return SPEC_ERR_UNSUPPORTED;
    if (rows == 0) return SPEC_OK;
    if (!hidden || !lm_head || !logits_out || !dev_status) return SPEC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15) || (reinterpret_cast<uintptr_t>(lm_head) & 15) ||
        (reinterpret_cast<uintptr_t>(logits_out) & 15))
        return SPEC_ERR_UNSUPPORTED;
    CUtensorMap ma, mb;
    spec_status st = make_map(&ma, hidden, rows, H, LM_BM);
    if (st != SPEC_OK) return st;
    st = make_map(&mb, lm_head, V, H, LM_BN);
    if (st != SPEC_OK) return st;
    if (lm_prepare() != SPEC_OK) return SPEC_ERR_CUDA;
    LmArgs L;
    L.rows = rows;
    L.H = H;
    L.V = V;
    L.out = static_cast<uint16_t*>(logits_out);
    L.status = dev_status;
    Params P = {};
    const dim3 grid(unsigned(row_tiles(rows)), unsigned((V + TILE - 1) / TILE));
    if (launch_lm<false>(grid, reinterpret_cast<cudaStream_t>(stream), ma, mb, L, P) !=
        cudaSuccess)
        return SPEC_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"
