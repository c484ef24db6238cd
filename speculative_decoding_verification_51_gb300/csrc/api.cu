// api.cu -- the C ABI declared in include/spec_verify.h: argument checks,
// workspace carving and the launch sequence of one verification call.
#include <cfloat>
#include <mutex>

#include "common.cuh"

using namespace sv;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int sms = 0;
    int stats_blocks_bf16 = 0;  // resident k_row_stats CTAs per SM
    int stats_blocks_f32 = 0;
    int sample_blocks_bf16 = 0;  // resident k_sample CTAs per SM
    int sample_blocks_f32 = 0;
    bool verify_bf16 = false;    // one k_verify CTA fits an SM
    bool verify_f32 = false;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

constexpr size_t stats_smem(int dtype) {
    return size_t(STATS_WARPS) * STATS_STAGES * TILE * (dtype == SPEC_BF16 ? 2 : 4);
}
// k_sample: SAMPLE_STAGES stages per warp pair of (logits chunk + draft-probability chunk)
constexpr size_t sample_smem(int dtype) {
    return size_t(SAMPLE_PAIRS) * SAMPLE_STAGES * TILE * ((dtype == SPEC_BF16 ? 2 : 4) + 4);
}
// k_emit: one such stage per warp
constexpr size_t emit_smem(int dtype) {
    return size_t(EMIT_WARPS) * TILE * ((dtype == SPEC_BF16 ? 2 : 4) + 4);
}

// Per-device launch facts, computed once per device (thread-safe).
spec_status device_info(DeviceInfo& out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SPEC_ERR_CUDA;
        if (cudaFuncSetAttribute(k_row_stats_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(stats_smem(SPEC_BF16))) != cudaSuccess ||
            cudaFuncSetAttribute(k_row_stats_f32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(stats_smem(SPEC_F32))) != cudaSuccess ||
            cudaFuncSetAttribute(k_sample_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sample_smem(SPEC_BF16))) != cudaSuccess ||
            cudaFuncSetAttribute(k_sample_f32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sample_smem(SPEC_F32))) != cudaSuccess ||
            cudaFuncSetAttribute(k_emit_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(emit_smem(SPEC_BF16))) != cudaSuccess ||
            cudaFuncSetAttribute(k_emit_f32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(emit_smem(SPEC_F32))) != cudaSuccess)
            return SPEC_ERR_CUDA;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.stats_blocks_bf16,
                                                          k_row_stats_bf16, STATS_WARPS * 32,
                                                          stats_smem(SPEC_BF16)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.stats_blocks_f32,
                                                          k_row_stats_f32, STATS_WARPS * 32,
                                                          stats_smem(SPEC_F32)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.sample_blocks_bf16, k_sample_bf16,
                                                          SAMPLE_PAIRS * 64,
                                                          sample_smem(SPEC_BF16)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.sample_blocks_f32, k_sample_f32,
                                                          SAMPLE_PAIRS * 64,
                                                          sample_smem(SPEC_F32)) != cudaSuccess)
            return SPEC_ERR_CUDA;
        int vb = 0, vf = 0;
        if (cudaFuncSetAttribute(k_verify_bf16, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(verify_smem(SPEC_BF16))) != cudaSuccess ||
            cudaFuncSetAttribute(k_verify_f32, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(verify_smem(SPEC_F32))) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&vb, k_verify_bf16,
                                                          verify_threads(SPEC_BF16),
                                                          verify_smem(SPEC_BF16)) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&vf, k_verify_f32,
                                                          verify_threads(SPEC_F32),
                                                          verify_smem(SPEC_F32)) != cudaSuccess)
            return SPEC_ERR_CUDA;
        d.verify_bf16 = vb >= 1;
        d.verify_f32 = vf >= 1;
        d.stats_blocks_bf16 = d.stats_blocks_bf16 < 1 ? 1 : d.stats_blocks_bf16;
        d.stats_blocks_f32 = d.stats_blocks_f32 < 1 ? 1 : d.stats_blocks_f32;
        d.sample_blocks_bf16 = d.sample_blocks_bf16 < 1 ? 1 : d.sample_blocks_bf16;
        d.sample_blocks_f32 = d.sample_blocks_f32 < 1 ? 1 : d.sample_blocks_f32;
        d.ready = true;
    }
    out = d;
    return SPEC_OK;
}

// Programmatic dependent launch lets a kernel's launch and prologue overlap
// its predecessor's tail; every kernel still executes griddepcontrol.wait
// before it reads its predecessor's output, so either launch mode is correct.
// Measured on GB300 for the all-rows pass (ms per call, plain order / PDL):
// direct launches 0.0354 / 0.0285 (B=1), 0.0648 / 0.0563 (B=64, V=128256),
// 0.0844 / 0.0740 (B=128, K=8); replays of a CUDA graph 0.0274 / 0.0287,
// 0.0574 / 0.0561, 0.0746 / 0.0728.  On unless -DSV_NO_PDL.
#ifdef SV_NO_PDL
constexpr bool kUsePdl = false;
#else
constexpr bool kUsePdl = true;
#endif
// Launches that use programmatic dependent launch even under SV_NO_PDL (bit
// 0 k_row_stats, 1 k_accept_all, 2 k_sample, 3 k_emit, 4 k_verify).
#ifndef SV_PDL_MASK
#define SV_PDL_MASK 16
#endif
constexpr unsigned kPdlMask = SV_PDL_MASK;

// Which verifier a lossless call runs: the caller's choice, or (PATH_AUTO)
// the faster one for the batch.  The request-by-request kernel gives each
// request one CTA, so it leaves SMs idle while B is small against the SM
// count and each CTA's rows are read one after another; the all-rows pass
// spreads every row over the whole GPU.  Measured on GB300 (152 SMs, bf16,
// CUDA-graph replays, ms per call, by request / all rows): K = 8, V = 129280:
// B = 256 0.1146 / 0.1099, B = 320 0.1290 / 0.1299, B = 384 0.1396 / 0.1527,
// B = 512 0.1608 / 0.1961; K = 3, V = 151936, B = 256: 0.0791 / 0.0776.
// Request by request from B of about 2.1 x the SM count.
enum { PATH_AUTO = 0, PATH_ALL_ROWS = 1, PATH_BY_REQUEST = 2 };
bool by_request_pays(long long B, int sms) { return 10 * B >= 21LL * sms; }

cudaError_t launch(void (*kern)(Params), unsigned grid, unsigned block, size_t smem,
                   cudaStream_t st, bool pdl, const Params& P, unsigned pdl_bit = 0) {
    pdl = pdl && (kUsePdl || (kPdlMask & pdl_bit));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

bool sizes_ok(int B, int K, int V) {
    return B >= 0 && B <= (1 << 24) && K >= 0 && K <= SPEC_MAX_K && V >= 8 && V <= (1 << 24);
}

template <typename T>
T* at(void* base, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

}  // namespace

static spec_status verify_impl(const void* target_logits, spec_dtype logits_dtype,
                           const float* draft_probs, const int32_t* draft_ids,
                           const int32_t* num_draft, const float* temperature, uint64_t seed,
                           int B, int K, int V, int32_t* out_ids, int32_t* out_num_accepted,
                           void* workspace, size_t workspace_bytes, spec_stream_t stream,
                           uint32_t request_offset, float* dbg_rows, float* dbg_req,
                           int32_t* dev_status, cudaEvent_t* events, int rule = RULE_LOSSLESS,
                           float threshold = 0.f, const int32_t* parents = nullptr,
                           int32_t* out_last = nullptr, const uint64_t* seed_dev = nullptr,
                           bool early_exit = false, const LmHeadIn* lm = nullptr,
                           const float* host_probs = nullptr, int path = PATH_AUTO) {
    const bool tree = parents != nullptr;
    if (!sizes_ok(B, K, V)) return SPEC_ERR_INVALID_ARG;
    if (rule == RULE_TYPICAL && threshold != threshold) return SPEC_ERR_INVALID_ARG;
    if (logits_dtype != SPEC_F32 && logits_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (V % 8 != 0) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!target_logits || !num_draft || !temperature || !out_ids || !out_num_accepted ||
        !workspace || (K > 0 && !draft_ids))
        return SPEC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(target_logits) & 15) ||
        (reinterpret_cast<uintptr_t>(draft_probs) & 15))
        return SPEC_ERR_UNSUPPORTED;
    const Layout L = make_layout(B, K, V);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255) || workspace_bytes < L.total)
        return SPEC_ERR_WORKSPACE;

    DeviceInfo dev;
    if (device_info(dev) != SPEC_OK) return SPEC_ERR_CUDA;

    Params P;
    P.logits = target_logits;
    P.probs = draft_probs;
    P.ids = draft_ids;
    P.num_draft = num_draft;
    P.temp = temperature;
    P.out_ids = out_ids;
    P.out_nacc = out_num_accepted;
    P.dbg_rows = dbg_rows;
    P.dbg_req = dbg_req;
    P.hdr = at<int>(workspace, L.hdr);
    P.status = dev_status ? dev_status : P.hdr + HDR_STATUS;
    P.rowlist = at<int>(workspace, L.rowlist);
    P.req_flags = at<int>(workspace, L.req_flags);
    P.part = at<Partial>(workspace, L.part);
    P.res_rec = at<ReqRec>(workspace, L.res_rec);
    P.bonus_rec = at<ReqRec>(workspace, L.bonus_rec);
    P.rsum = at<float>(workspace, L.rsum);
    P.gath = at<float2>(workspace, L.gath);
    P.cnt = at<int>(workspace, L.cnt);
    P.round = early_exit ? 0 : -1;
    P.tree = tree ? 1 : 0;
    P.parents = parents;
    P.out_last = out_last;
    P.tmass = at<float>(workspace, L.tmass);
    P.seed = seed;
    P.seed_dev = seed_dev;
    P.req_off = request_offset;
    P.rule = rule;
    P.threshold = threshold;
    P.dtype = logits_dtype;
    P.B = B;
    P.K = K;
    P.K1 = K + 1;
    P.V = V;
    P.C = (V + TILE - 1) / TILE;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const bool bf16 = logits_dtype == SPEC_BF16;
    // events (profiling only) are recorded before each kernel and after the last
    auto mark = [&](int i) { return events ? cudaEventRecord(events[i], st) : cudaSuccess; };

    // The request-by-request verifier (verify.cu): every lossless call whose
    // rows fit its tile buffers, unless the caller asks for the all-rows pass.
    const bool fits = !tree && !early_exit && !lm && !host_probs && rule == RULE_LOSSLESS &&
                      P.C <= VCMAX && (bf16 ? dev.verify_bf16 : dev.verify_f32);
    const bool by_request = fits && path != PATH_ALL_ROWS &&
                            (path == PATH_BY_REQUEST || by_request_pays(B, dev.sms));
    if (by_request) {
        const long long gv = B < dev.sms ? B : dev.sms;
        cudaError_t e = mark(0);
        if (e == cudaSuccess) e = launch(k_prep, 1, 1024, 0, st, false, P);
        if (e == cudaSuccess) e = mark(1);
        if (e == cudaSuccess)
            e = launch(bf16 ? k_verify_bf16 : k_verify_f32, unsigned(gv),
                       unsigned(verify_threads(logits_dtype)), verify_smem(logits_dtype), st,
                       true, P, 16u);
        for (int i = 2; i <= 5 && e == cudaSuccess; ++i) e = mark(i);
        return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
    }

    const long long max_tiles = (long long)B * P.K1 * P.C;
    long long g1 = (long long)dev.sms * (bf16 ? dev.stats_blocks_bf16 : dev.stats_blocks_f32);
    const long long need1 = (max_tiles + STATS_WARPS - 1) / STATS_WARPS;
    if (g1 > need1) g1 = need1;
    long long g3 = (long long)dev.sms * (bf16 ? dev.sample_blocks_bf16 : dev.sample_blocks_f32);
    const long long need3 = ((long long)B * P.C + SAMPLE_PAIRS - 1) / SAMPLE_PAIRS;
    if (g3 > need3) g3 = need3;
    // k_emit: a warp per slot of the residual and of the bonus queue
    const unsigned g4 = unsigned((2LL * B + EMIT_WARPS - 1) / EMIT_WARPS);

    cudaError_t e = mark(0);
    if (e == cudaSuccess) e = launch(k_plan, 1, PLAN_THREADS, 0, st, false, P);
    if (e == cudaSuccess) e = mark(1);
    if (lm) {
        // the logits are produced here, with their row statistics and acceptances
        if (e == cudaSuccess && launch_lmhead_fused(P, *lm, st) != SPEC_OK) return SPEC_ERR_CUDA;
    } else if (early_exit) {
        // one pass per draft position: pass r reads row r of the requests that
        // kept drafts 0..r-1; a request leaves at its first rejection
        long long gr = (long long)dev.sms * (bf16 ? dev.stats_blocks_bf16 : dev.stats_blocks_f32);
        const long long need = ((long long)B * P.C + STATS_WARPS - 1) / STATS_WARPS;
        if (gr > need) gr = need;
        for (int r = 0; r <= K && e == cudaSuccess; ++r) {
            P.round = r;
            e = launch(bf16 ? k_row_stats_bf16 : k_row_stats_f32, unsigned(gr), STATS_WARPS * 32,
                       stats_smem(logits_dtype), st, true, P);
        }
    } else if (e == cudaSuccess) {
        e = launch(bf16 ? k_row_stats_bf16 : k_row_stats_f32, unsigned(g1),
                   STATS_WARPS * 32, stats_smem(logits_dtype), st, true, P, 1u);
    }
    if (e == cudaSuccess) e = mark(2);
    if (tree) {  // the walks, one CTA per request
        if (e == cudaSuccess)
            e = launch(bf16 ? k_tree_walk_bf16 : k_tree_walk_f32, unsigned(B), TREE_THREADS, 0,
                       st, false, P);
        return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
    }
    // the all-rows pass leaves the acceptances to one warp per request here
    if (!lm && !early_exit && e == cudaSuccess)
        e = launch(k_accept_all, unsigned(B), ACCEPT_WARPS * 32, 0, st, true, P, 2u);
    // spec_verify_host: the q rows of the residual draws, now that they are known
    if (host_probs && e == cudaSuccess) {
        const long long g = B < 4LL * dev.sms ? B : 4LL * dev.sms;
        k_qrows_in<<<unsigned(g > 0 ? g : 1), HOST_IO_THREADS, 0, st>>>(P, host_probs);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = mark(3);
    // typical acceptance draws every token from p, and without draft
    // distributions no request can take a residual draw: no k_sample then
    const bool residuals = rule != RULE_TYPICAL && P.probs != nullptr;
    if (e == cudaSuccess && residuals)
        e = launch(bf16 ? k_sample_bf16 : k_sample_f32, unsigned(g3), SAMPLE_PAIRS * 64,
                   sample_smem(logits_dtype), st, true, P, 4u);
    if (e == cudaSuccess) e = mark(4);
    if (e == cudaSuccess)
        e = launch(bf16 ? k_emit_bf16 : k_emit_f32, g4, EMIT_WARPS * 32,
                   emit_smem(logits_dtype), st, true, P, 8u);
    if (e == cudaSuccess) e = mark(5);
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" {

const char* spec_status_str(spec_status s) {
    switch (s) {
        case SPEC_OK: return "SPEC_OK";
        case SPEC_ERR_INVALID_ARG: return "SPEC_ERR_INVALID_ARG";
        case SPEC_ERR_UNSUPPORTED: return "SPEC_ERR_UNSUPPORTED";
        case SPEC_ERR_CUDA: return "SPEC_ERR_CUDA";
        case SPEC_ERR_WORKSPACE: return "SPEC_ERR_WORKSPACE";
    }
    return "SPEC_ERR_UNKNOWN";
}

size_t spec_verify_workspace_size(int B, int K, int V) {
    if (!sizes_ok(B, K, V) || V % 8 != 0) return 0;
    return make_layout(B, K, V).total;
}

int32_t* spec_verify_status_ptr(void* workspace) {
    return workspace ? at<int32_t>(workspace, 0) + HDR_STATUS : nullptr;
}

spec_status spec_verify_ex(const void* target_logits, spec_dtype logits_dtype,
                           const float* draft_probs, const int32_t* draft_ids,
                           const int32_t* num_draft, const float* temperature, uint64_t seed,
                           int B, int K, int V, int32_t* out_ids, int32_t* out_num_accepted,
                           void* workspace, size_t workspace_bytes, spec_stream_t stream,
                           uint32_t request_offset, float* dbg_rows, float* dbg_req,
                           int32_t* dev_status) {
    return verify_impl(target_logits, logits_dtype, draft_probs, draft_ids, num_draft,
                       temperature, seed, B, K, V, out_ids, out_num_accepted, workspace,
                       workspace_bytes, stream, request_offset, dbg_rows, dbg_req, dev_status,
                       nullptr);
}

spec_status spec_verify_typical(const void* target_logits, spec_dtype logits_dtype,
                                const int32_t* draft_ids, const int32_t* num_draft,
                                const float* temperature, float threshold, uint64_t seed, int B,
                                int K, int V, int32_t* out_ids, int32_t* out_num_accepted,
                                void* workspace, size_t workspace_bytes, spec_stream_t stream,
                                uint32_t request_offset, float* dbg_rows, float* dbg_req,
                                int32_t* dev_status) {
    return verify_impl(target_logits, logits_dtype, nullptr, draft_ids, num_draft, temperature,
                       seed, B, K, V, out_ids, out_num_accepted, workspace, workspace_bytes,
                       stream, request_offset, dbg_rows, dbg_req, dev_status, nullptr,
                       RULE_TYPICAL, threshold);
}

spec_status spec_verify_dev_seed(const void* target_logits, spec_dtype logits_dtype,
                                 const float* draft_probs, const int32_t* draft_ids,
                                 const int32_t* num_draft, const float* temperature,
                                 const uint64_t* seed_dev, int B, int K, int V, int32_t* out_ids,
                                 int32_t* out_num_accepted, void* workspace,
                                 size_t workspace_bytes, spec_stream_t stream,
                                 uint32_t request_offset, float* dbg_rows, float* dbg_req,
                                 int32_t* dev_status) {
    if (!seed_dev || (reinterpret_cast<uintptr_t>(seed_dev) & 7)) return SPEC_ERR_INVALID_ARG;
    return verify_impl(target_logits, logits_dtype, draft_probs, draft_ids, num_draft,
                       temperature, 0, B, K, V, out_ids, out_num_accepted, workspace,
                       workspace_bytes, stream, request_offset, dbg_rows, dbg_req, dev_status,
                       nullptr, RULE_LOSSLESS, 0.f, nullptr, nullptr, seed_dev);
}

spec_status spec_verify_early_exit(const void* target_logits, spec_dtype logits_dtype,
                                   const float* draft_probs, const int32_t* draft_ids,
                                   const int32_t* num_draft, const float* temperature,
                                   uint64_t seed, int B, int K, int V, int32_t* out_ids,
                                   int32_t* out_num_accepted, void* workspace,
                                   size_t workspace_bytes, spec_stream_t stream,
                                   uint32_t request_offset, float* dbg_rows, float* dbg_req,
                                   int32_t* dev_status, const uint64_t* seed_dev) {
    if (reinterpret_cast<uintptr_t>(seed_dev) & 7) return SPEC_ERR_INVALID_ARG;
    return verify_impl(target_logits, logits_dtype, draft_probs, draft_ids, num_draft,
                       temperature, seed, B, K, V, out_ids, out_num_accepted, workspace,
                       workspace_bytes, stream, request_offset, dbg_rows, dbg_req, dev_status,
                       nullptr, RULE_LOSSLESS, 0.f, nullptr, nullptr, seed_dev, true);
}

spec_status spec_verify_all_rows(const void* target_logits, spec_dtype logits_dtype,
                                 const float* draft_probs, const int32_t* draft_ids,
                                 const int32_t* num_draft, const float* temperature,
                                 uint64_t seed, int B, int K, int V, int32_t* out_ids,
                                 int32_t* out_num_accepted, void* workspace,
                                 size_t workspace_bytes, spec_stream_t stream,
                                 uint32_t request_offset, float* dbg_rows, float* dbg_req,
                                 int32_t* dev_status, const uint64_t* seed_dev,
                                 spec_event_t* events) {
    if (reinterpret_cast<uintptr_t>(seed_dev) & 7) return SPEC_ERR_INVALID_ARG;
    if (events)
        for (int i = 0; i < 6; ++i)
            if (!events[i]) return SPEC_ERR_INVALID_ARG;
    return verify_impl(target_logits, logits_dtype, draft_probs, draft_ids, num_draft,
                       temperature, seed, B, K, V, out_ids, out_num_accepted, workspace,
                       workspace_bytes, stream, request_offset, dbg_rows, dbg_req, dev_status,
                       reinterpret_cast<cudaEvent_t*>(events), RULE_LOSSLESS, 0.f, nullptr,
                       nullptr, seed_dev, false, nullptr, nullptr, PATH_ALL_ROWS);
}

spec_status spec_verify_by_request(const void* target_logits, spec_dtype logits_dtype,
                                   const float* draft_probs, const int32_t* draft_ids,
                                   const int32_t* num_draft, const float* temperature,
                                   uint64_t seed, int B, int K, int V, int32_t* out_ids,
                                   int32_t* out_num_accepted, void* workspace,
                                   size_t workspace_bytes, spec_stream_t stream,
                                   uint32_t request_offset, float* dbg_rows, float* dbg_req,
                                   int32_t* dev_status, const uint64_t* seed_dev,
                                   spec_event_t* events) {
    if (reinterpret_cast<uintptr_t>(seed_dev) & 7) return SPEC_ERR_INVALID_ARG;
    if (events)
        for (int i = 0; i < 6; ++i)
            if (!events[i]) return SPEC_ERR_INVALID_ARG;
    return verify_impl(target_logits, logits_dtype, draft_probs, draft_ids, num_draft,
                       temperature, seed, B, K, V, out_ids, out_num_accepted, workspace,
                       workspace_bytes, stream, request_offset, dbg_rows, dbg_req, dev_status,
                       reinterpret_cast<cudaEvent_t*>(events), RULE_LOSSLESS, 0.f, nullptr,
                       nullptr, seed_dev, false, nullptr, nullptr, PATH_BY_REQUEST);
}

int spec_verify_path(int B, int K, int V, spec_dtype logits_dtype) {
    if (!sizes_ok(B, K, V) || V % 8 != 0) return -1;
    if (logits_dtype != SPEC_F32 && logits_dtype != SPEC_BF16) return -1;
    DeviceInfo dev;
    if (device_info(dev) != SPEC_OK) return -1;
    const bool fits = (V + TILE - 1) / TILE <= VCMAX &&
                      (logits_dtype == SPEC_BF16 ? dev.verify_bf16 : dev.verify_f32);
    return fits && by_request_pays(B, dev.sms) ? 1 : 0;
}

size_t spec_verify_lmhead_workspace_size(int B, int K, int V, int H) {
    if (!sizes_ok(B, K, V) || V % 8 != 0 || H <= 0 || H % 64 != 0 || H > (1 << 16)) return 0;
    return make_layout(B, K, V).total + align256(size_t(B) * (K + 1) * H * 2);
}

spec_status spec_verify_lmhead(const void* hidden, const void* lm_head, int H, void* logits_out,
                               const float* draft_probs, const int32_t* draft_ids,
                               const int32_t* num_draft, const float* temperature, uint64_t seed,
                               int B, int K, int V, int32_t* out_ids, int32_t* out_num_accepted,
                               void* workspace, size_t workspace_bytes, spec_stream_t stream,
                               uint32_t request_offset, float* dbg_rows, float* dbg_req,
                               int32_t* dev_status) {
    if (!sizes_ok(B, K, V) || H <= 0 || H > (1 << 16)) return SPEC_ERR_INVALID_ARG;
    if (H % 64 != 0 || V % 8 != 0) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!hidden || !lm_head || !logits_out) return SPEC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15) || (reinterpret_cast<uintptr_t>(lm_head) & 15))
        return SPEC_ERR_UNSUPPORTED;
    const size_t base = make_layout(B, K, V).total;
    if (workspace_bytes < spec_verify_lmhead_workspace_size(B, K, V, H)) return SPEC_ERR_WORKSPACE;
    LmHeadIn in;
    in.hidden = hidden;
    in.lm_head = lm_head;
    in.H = H;
    in.hid_c = static_cast<char*>(workspace) + base;
    return verify_impl(logits_out, SPEC_BF16, draft_probs, draft_ids, num_draft, temperature, seed,
                       B, K, V, out_ids, out_num_accepted, workspace, workspace_bytes, stream,
                       request_offset, dbg_rows, dbg_req, dev_status, nullptr, RULE_LOSSLESS, 0.f,
                       nullptr, nullptr, nullptr, false, &in);
}

size_t spec_verify_tree_workspace_size(int B, int N, int V) {
    if (N < 1 || N > TREE_MAX_NODES) return 0;
    return spec_verify_workspace_size(B, N - 1, V);
}

spec_status spec_verify_tree(const void* target_logits, spec_dtype logits_dtype,
                             const float* draft_probs, const int32_t* tree_tokens,
                             const int32_t* tree_parents, const int32_t* num_nodes,
                             const float* temperature, uint64_t seed, int B, int N, int V,
                             int32_t* out_ids, int32_t* out_num_accepted,
                             int32_t* out_last_node, void* workspace, size_t workspace_bytes,
                             spec_stream_t stream, uint32_t request_offset, float* dbg_nodes,
                             float* dbg_req, int32_t* dev_status) {
    if (N < 1) return SPEC_ERR_INVALID_ARG;
    if (N > TREE_MAX_NODES) return SPEC_ERR_UNSUPPORTED;
    if (B > 0 && (!tree_tokens || !tree_parents || !out_last_node)) return SPEC_ERR_INVALID_ARG;
    return verify_impl(target_logits, logits_dtype, draft_probs, tree_tokens, num_nodes,
                       temperature, seed, B, N - 1, V, out_ids, out_num_accepted, workspace,
                       workspace_bytes, stream, request_offset, dbg_nodes, dbg_req, dev_status,
                       nullptr, RULE_LOSSLESS, 0.f, tree_parents, out_last_node);
}

spec_status spec_verify_profiled(const void* target_logits, spec_dtype logits_dtype,
                                 const float* draft_probs, const int32_t* draft_ids,
                                 const int32_t* num_draft, const float* temperature,
                                 uint64_t seed, int B, int K, int V, int32_t* out_ids,
                                 int32_t* out_num_accepted, void* workspace,
                                 size_t workspace_bytes, spec_stream_t stream,
                                 spec_event_t* events) {
    if (!events) return SPEC_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (!events[i]) return SPEC_ERR_INVALID_ARG;
    return verify_impl(target_logits, logits_dtype, draft_probs, draft_ids, num_draft,
                       temperature, seed, B, K, V, out_ids, out_num_accepted, workspace,
                       workspace_bytes, stream, 0u, nullptr, nullptr, nullptr,
                       reinterpret_cast<cudaEvent_t*>(events));
}

spec_status spec_verify(const void* target_logits, spec_dtype logits_dtype,
                        const float* draft_probs, const int32_t* draft_ids,
                        const int32_t* num_draft, const float* temperature, uint64_t seed, int B,
                        int K, int V, int32_t* out_ids, int32_t* out_num_accepted,
                        void* workspace, size_t workspace_bytes, spec_stream_t stream) {
    return spec_verify_ex(target_logits, logits_dtype, draft_probs, draft_ids, num_draft,
                          temperature, seed, B, K, V, out_ids, out_num_accepted, workspace,
                          workspace_bytes, stream, 0u, nullptr, nullptr, nullptr);
}

// The device address of a page-locked host buffer mapped into the device's
// address space, or nullptr for any other memory.
static const void* mapped_device_ptr(const void* h) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, h) != cudaSuccess) {
        (void)cudaGetLastError();  // not a pointer CUDA knows
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// Small device buffer of spec_verify_host: ids, num_draft, temperature,
// out_ids, out_num_accepted, each 256-byte aligned.
size_t spec_verify_host_small_bytes(int B, int K) {
    if (B < 0 || K < 0 || K > SPEC_MAX_K) return 0;
    const size_t b = size_t(B), k1 = size_t(K) + 1;
    return align256(b * K * 4) + align256(b * 4) + align256(b * 4) + align256(b * k1 * 4) +
           align256(b * 4);
}

spec_status spec_verify_host(const void* h_logits, spec_dtype logits_dtype, const float* h_probs,
                             const int32_t* h_draft_ids, const int32_t* h_num_draft,
                             const float* h_temperature, uint64_t seed, int B, int K, int V,
                             int32_t* h_out_ids, int32_t* h_out_num_accepted, void* d_logits,
                             float* d_probs, void* d_small, void* workspace,
                             size_t workspace_bytes, spec_stream_t stream) {
    if (!sizes_ok(B, K, V)) return SPEC_ERR_INVALID_ARG;
    if (logits_dtype != SPEC_F32 && logits_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
    if (V % 8 != 0) return SPEC_ERR_UNSUPPORTED;
    if (B == 0) return SPEC_OK;
    if (!h_logits || !h_num_draft || !h_temperature || !h_out_ids || !h_out_num_accepted ||
        !d_logits || !d_small || (K > 0 && !h_draft_ids) || (h_probs && !d_probs))
        return SPEC_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(d_small) & 255) return SPEC_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const size_t b = size_t(B), k1 = size_t(K) + 1, esz = logits_dtype == SPEC_BF16 ? 2 : 4;
    char* s = static_cast<char*>(d_small);
    int32_t* d_ids = reinterpret_cast<int32_t*>(s);
    s += align256(b * K * 4);
    int32_t* d_num = reinterpret_cast<int32_t*>(s);
    s += align256(b * 4);
    float* d_temp = reinterpret_cast<float*>(s);
    s += align256(b * 4);
    int32_t* d_out = reinterpret_cast<int32_t*>(s);
    s += align256(b * k1 * 4);
    int32_t* d_nacc = reinterpret_cast<int32_t*>(s);

    // Page-locked host buffers mapped into the device's address space are read
    // by copy kernels, and only what the verifier reads crosses the link: the
    // logits rows 0..n_b, q_j(x_j), and the q rows of the residual draws.
    // Other host memory takes whole-tensor copies.
    const void* m_logits = mapped_device_ptr(h_logits);
    const float* m_probs = h_probs ? static_cast<const float*>(mapped_device_ptr(h_probs)) : nullptr;
    const bool rows_only = m_logits && (!h_probs || m_probs);
    cudaError_t e = cudaSuccess;
    if (K > 0) e = cudaMemcpyAsync(d_ids, h_draft_ids, b * K * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_num, h_num_draft, b * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_temp, h_temperature, b * 4, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && rows_only) {
        DeviceInfo dev;
        if (device_info(dev) != SPEC_OK) return SPEC_ERR_CUDA;
        const long long rows = (long long)B * k1;
        const long long g = rows < 16LL * dev.sms ? rows : 16LL * dev.sms;
        k_rows_in<<<unsigned(g), HOST_IO_THREADS, 0, st>>>(m_logits, d_logits, d_num, B, K,
                                                           size_t(V) * esz);
        e = cudaGetLastError();
        if (e == cudaSuccess && h_probs && K > 0) {
            k_qx_in<<<unsigned(B), 32, 0, st>>>(m_probs, d_probs, d_ids, d_num, B, K, V);
            e = cudaGetLastError();
        }
    } else if (e == cudaSuccess) {
        e = cudaMemcpyAsync(d_logits, h_logits, b * k1 * V * esz, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess && h_probs)
            e = cudaMemcpyAsync(d_probs, h_probs, b * K * V * 4, cudaMemcpyHostToDevice, st);
    }
    if (e != cudaSuccess) return SPEC_ERR_CUDA;
    const spec_status r = verify_impl(
        d_logits, logits_dtype, h_probs ? d_probs : nullptr, K > 0 ? d_ids : nullptr, d_num, d_temp,
        seed, B, K, V, d_out, d_nacc, workspace, workspace_bytes, stream, 0, nullptr, nullptr,
        nullptr, nullptr, RULE_LOSSLESS, 0.f, nullptr, nullptr, nullptr, false, nullptr,
        rows_only ? m_probs : nullptr);
    if (r != SPEC_OK) return r;
    e = cudaMemcpyAsync(h_out_ids, d_out, b * k1 * 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(h_out_num_accepted, d_nacc, b * 4, cudaMemcpyDeviceToHost, st);
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// spec_verify_noalloc: spec_verify for callers that cannot allocate device
// memory.  Its scratch is the file-scope array below, created with the module
// on every GPU that loads this library and kept until the process exits.
// Host code only ever sees a host-side stand-in for the array's name, so the
// device address is looked up once per device (cudaGetSymbolAddress, with
// that device current) on the first call made on that device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[kMaxDevices] = {};

static spec_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SPEC_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return SPEC_OK;
}

spec_status spec_verify_noalloc(const void* target_logits, spec_dtype logits_dtype,
                                const float* draft_probs, const int32_t* draft_ids,
                                const int32_t* num_draft, const float* temperature, uint64_t seed,
                                int B, int K, int V, int32_t* out_ids, int32_t* out_num_accepted,
                                spec_stream_t stream) {
    if (!sizes_ok(B, K, V)) return SPEC_ERR_INVALID_ARG;
    if (V % 8 != 0) return SPEC_ERR_UNSUPPORTED;
    if (make_layout(B, K, V).total > SPEC_NOALLOC_SCRATCH_BYTES) return SPEC_ERR_WORKSPACE;
    void* scratch = nullptr;
    const spec_status s = noalloc_scratch(&scratch);
    if (s != SPEC_OK) return s;
    return spec_verify(target_logits, logits_dtype, draft_probs, draft_ids, num_draft,
                       temperature, seed, B, K, V, out_ids, out_num_accepted, scratch,
                       SPEC_NOALLOC_SCRATCH_BYTES, stream);
}

spec_status spec_philox_fill(uint64_t seed, const uint32_t* ctrs, int64_t n, uint32_t* out,
                             spec_stream_t stream) {
    if (n < 0 || (n > 0 && (!ctrs || !out))) return SPEC_ERR_INVALID_ARG;
    if (n == 0) return SPEC_OK;
    const long long blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    k_philox_fill<<<unsigned(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(seed, ctrs,
                                                                                      n, out);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"

namespace sv {
__global__ void k_philox_fill(uint64_t seed, const uint32_t* ctrs, int64_t n, uint32_t* out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 c = reinterpret_cast<const uint4*>(ctrs)[i];
        reinterpret_cast<uint4*>(out)[i] = philox4x32_10(c, uint32_t(seed), uint32_t(seed >> 32));
    }
}
}  // namespace sv
