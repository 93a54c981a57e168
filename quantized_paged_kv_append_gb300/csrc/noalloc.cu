// noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// kv_decode_attn needs a caller-provided workspace (split-K partial results and
// merge records). Some callers have no way to provide one: code that runs
// while a stream is being captured into a CUDA graph (device allocation is not
// allowed there), hosts whose device memory belongs entirely to another pool or
// framework, and latency-critical loops that must never allocate. For them this
// file keeps a fixed scratch area in static device memory and runs the same
// decode kernel on it. Every GPU that loads the library reserves this area
// until the process exits.
#include <cstdint>
#include <mutex>

#include "../../include/qkv.h"
#include "qkv_device.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB, shared by every call on a device

static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDev];   // device address of g_decode_scratch, per device

// Resolves the scratch array's device address for the current device (once).
int scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDev) return QKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr) return QKV_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return QKV_OK;
}

}  // namespace

extern "C" int kv_decode_attn_noalloc(const qkv_cache_desc* cache, const void* q, const void* k_new, const void* v_new,
                                      int batch, int num_q_heads, const int32_t* page_table, int max_pages_per_seq,
                                      const int32_t* seq_lens, int max_seq_len, float scale, void* out, int out_dtype,
                                      void* stream) {
    if (batch == 0) return kv_decode_attn(cache, q, k_new, v_new, 0, num_q_heads, page_table, max_pages_per_seq,
                                          seq_lens, max_seq_len, scale, out, out_dtype, nullptr, 0, stream);
    const size_t need = kv_decode_workspace_size(cache, batch, num_q_heads, max_seq_len);
    if (need == 0) {
        // invalid arguments: let the regular entry point report which one
        return kv_decode_attn(cache, q, k_new, v_new, batch, num_q_heads, page_table, max_pages_per_seq, seq_lens,
                              max_seq_len, scale, out, out_dtype, nullptr, 0, stream);
    }
    if (need > kNoAllocScratchBytes) return QKV_ERR_WORKSPACE;
    void* scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc) return rc;
    // The scratch keeps the previous call's contents. Every call writes its merge
    // records before the merge reads them, so nothing has to start at zero;
    // clearing the used span still keeps each call independent of whatever an
    // interrupted earlier call left there.
    if (cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream) != cudaSuccess) return QKV_ERR_CUDA;
    return kv_decode_attn(cache, q, k_new, v_new, batch, num_q_heads, page_table, max_pages_per_seq, seq_lens,
                          max_seq_len, scale, out, out_dtype, scratch, kNoAllocScratchBytes, stream);
}
