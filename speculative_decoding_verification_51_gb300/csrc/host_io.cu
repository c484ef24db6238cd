// host_io.cu -- the copy kernels of spec_verify_host when the caller's host
// buffers are page-locked and mapped into the device's address space: only
// the data the verifier reads crosses the host link.
//
//   k_rows_in   logits rows j = 0..n_b of every request (rows past num_draft
//               are never read; "投机采样" 第二步: one target pass scores
//               positions 1..gamma+1, of which a request uses n_b + 1);
//   k_qx_in     q_j(x_j) of every draft j < n_b (the acceptance ratio);
//   k_qrows_in  after the acceptances, the whole q row of the first
//               rejected position of each queued residual request (the only
//               q rows max(0, p - q) needs).
// Rows that are not copied keep whatever the device buffers held; no kernel
// of the call reads them.
#include "common.cuh"

namespace sv {

namespace {

// Copy `bytes` (a multiple of 16) from src to dst with the whole CTA.
__device__ __forceinline__ void copy_row(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                         size_t bytes) {
    const size_t n = bytes / 16;
    size_t i = threadIdx.x;
    for (; i + 3 * blockDim.x < n; i += 4 * blockDim.x) {
        const uint4 a = src[i], b = src[i + blockDim.x], c = src[i + 2 * blockDim.x],
                    d = src[i + 3 * blockDim.x];
        dst[i] = a;
        dst[i + blockDim.x] = b;
        dst[i + 2 * blockDim.x] = c;
        dst[i + 3 * blockDim.x] = d;
    }
    for (; i < n; i += blockDim.x) dst[i] = src[i];
}

// num_draft[b] clamped to the rows a request can have (a bad value copies
// row 0 only; the request is rejected as bad by k_plan)
__device__ __forceinline__ int rows_of(const int32_t* num, int b, int K) {
    const int n = num[b];
    return (n < 0 || n > K) ? 1 : n + 1;
}

}  // namespace

// grid: one CTA per (request b, row j), blockIdx.x = b * (K + 1) + j
__global__ void __launch_bounds__(HOST_IO_THREADS) k_rows_in(const void* src, void* dst,
                                                             const int32_t* num, int B, int K,
                                                             size_t row_bytes) {
    const int K1 = K + 1;
    for (long long r = blockIdx.x; r < (long long)B * K1; r += gridDim.x) {
        const int b = int(r / K1), j = int(r - (long long)b * K1);
        if (j >= rows_of(num, b, K)) continue;
        copy_row(reinterpret_cast<const uint4*>(static_cast<const char*>(src) + r * row_bytes),
                 reinterpret_cast<uint4*>(static_cast<char*>(dst) + r * row_bytes), row_bytes);
    }
}

// grid: one warp per request; lane j copies q_j(x_j) for j < n_b
__global__ void __launch_bounds__(32) k_qx_in(const float* src, float* dst, const int32_t* ids,
                                              const int32_t* num, int B, int K, int V) {
    const int b = blockIdx.x, j = threadIdx.x;
    if (b >= B) return;
    const int n = num[b];
    for (int jj = j; jj < K && jj < n; jj += 32) {
        const int x = ids[(size_t)b * K + jj];
        if (x < 0 || x >= V) continue;  // reported by the acceptance step
        const size_t e = ((size_t)b * K + jj) * V + x;
        dst[e] = src[e];
    }
}

// grid: one CTA per residual queue slot (after k_accept_all, before k_sample).
// P.probs is the caller's writable d_probs of spec_verify_host (the verifier
// itself only reads it, hence the const in Params).
__global__ void __launch_bounds__(HOST_IO_THREADS) k_qrows_in(Params P, const float* src) {
    const int n_res = P.hdr[HDR_NRES];
    for (int slot = blockIdx.x; slot < n_res; slot += gridDim.x) {
        const ReqRec r = P.res_rec[slot];
        const size_t off = ((size_t)r.b * P.K + r.erow) * P.V;
        copy_row(reinterpret_cast<const uint4*>(src + off),
                 reinterpret_cast<uint4*>(const_cast<float*>(P.probs) + off), size_t(P.V) * 4);
    }
}

}  // namespace sv
