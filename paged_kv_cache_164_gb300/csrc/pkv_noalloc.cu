// Decode attention without caller-provided workspace: the split-K partials go
// to a fixed array in the library's own device memory instead (see the
// declaration in pkv.h for who needs this and the rules that come with it).
#include <atomic>

#include "pkv_common.cuh"

namespace pkv {

// Reserved on every device that loads the library, for the life of the process.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static std::atomic<void*> g_scratch_address[kMaxDevices];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device.  In host code the array's name is only a host-side stand-in, so the
// real address must come from the runtime.
static pkv_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    void* ptr = g_scratch_address[dev].load(std::memory_order_acquire);
    if (ptr == nullptr) {
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return PKV_ERR_CUDA;
        }
        g_scratch_address[dev].store(ptr, std::memory_order_release);
    }
    *out = ptr;
    return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_decode_attention_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_blocks, int block_size, int num_q_heads,
    int num_kv_heads, int head_dim, float scale, int num_splits, pkv_dtype dtype,
    int32_t* err_flag, void* stream) {
    const size_t need = pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                  block_size, max_context_len, num_splits);
    if (need == SIZE_MAX) {
        // same argument checks and status as the workspace-taking call
        return pkv_decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                    context_lens, max_context_len, num_seqs, num_blocks,
                                    block_size, num_q_heads, num_kv_heads, head_dim, scale,
                                    num_splits, nullptr, 0, dtype, err_flag, stream);
    }
    if (need > PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (need > 0) {
        pkv_status st = scratch_address(&scratch);
        if (st != PKV_OK) return st;
    }
    return pkv_decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, max_context_len, num_seqs, num_blocks, block_size,
                                num_q_heads, num_kv_heads, head_dim, scale, num_splits, scratch,
                                need > 0 ? (size_t)PKV_NOALLOC_SCRATCH_BYTES : 0, dtype, err_flag,
                                stream);
}
