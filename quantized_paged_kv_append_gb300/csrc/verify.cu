// verify.cu -- the verify window: several decode queries per sequence, query j
// of a window of W at position seq_len - W + j, attending [0, seq_len - W + j + 1).
//
// Method (page title, section): "qwen35/q36: --kv - int8 K/V caches", "What it
// does" (the verify windows of speculative decoding go through the decode
// kernels); "--kv k8v4: hybrid KV cache", "Tests" (the batched forms with
// per-query step arrays).
//
// A small kernel expands the window into one decode row per query inside the
// caller's workspace: the sequence's page-table row is copied for every query
// and the query's own length is written beside it. The tensor-core decode then
// runs over the expanded rows unchanged (each query re-reads its prefix: W
// times the packed bytes of one decode step).
#include "qkv_device.cuh"
#include "qkv_params.h"

namespace qkv {

__device__ unsigned int g_err_verify;

// Block r: query row r. Its sequence b is found by a binary search of cu.
__global__ void __launch_bounds__(128) verify_expand_kernel(const VerifyParams p) {
    __shared__ int s_b;
    const int r = blockIdx.x;
    if (threadIdx.x == 0) {
        int lo = 0, hi = p.B - 1;   // the last b with cu[b] <= r
        if (p.cu) {
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (p.cu[mid] <= r) lo = mid;
                else hi = mid - 1;
            }
        } else {
            lo = r / p.W_fixed;     // windows of the same length: rows b W .. b W + W - 1
        }
        s_b = lo;
    }
    __syncthreads();
    const int b = s_b;
    const int c0 = p.cu ? p.cu[b] : b * p.W_fixed, W = p.cu ? p.cu[b + 1] - c0 : p.W_fixed, j = r - c0;
    int L = p.seq_lens[b];
    const int Lmax = p.max_pages * kPage;
    if (threadIdx.x == 0) {
        if (L < 0 || L > Lmax || W > L || j < 0 || j >= W) atomicOr(&g_err_verify, kErrPos);
    }
    L = max(0, min(L, Lmax));
    if (threadIdx.x == 0) p.lens_rep[r] = (j >= 0 && j < W) ? max(0, min(L, L - W + j + 1)) : 0;
    const int32_t* src = p.page_table + (size_t)b * p.max_pages;
    int32_t* dst = p.table_rep + (size_t)r * p.max_pages;
    for (int i = threadIdx.x; i < p.max_pages; i += blockDim.x) dst[i] = src[i];
}

cudaError_t verify_read_error(unsigned* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_err_verify, sizeof(unsigned));
    if (e != cudaSuccess || !clear) return e;
    unsigned z = 0;
    return cudaMemcpyToSymbol(g_err_verify, &z, sizeof(unsigned));
}

cudaError_t verify_expand_launch(const VerifyParams& p, int total_q, cudaStream_t st) {
    if (total_q <= 0) return cudaSuccess;
    verify_expand_kernel<<<total_q, 128, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace qkv
