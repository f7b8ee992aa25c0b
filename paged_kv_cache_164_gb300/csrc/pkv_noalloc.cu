// Decode attention without caller-provided workspace: the split-K partials go
// to a fixed array in the library's own device memory instead (see the
// declaration in pkv.h for who needs this and the rules that come with it).
#include <cudaTypedefs.h>

#include <mutex>

#include "pkv_common.cuh"

namespace pkv {

// Reserved on every device that loads the library, for the life of the process.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

// The array's device address differs from one CUDA context to the next (each
// context loads the library's device code on its own), so it is looked up
// once per context and remembered under the context's id.  cuCtxGetId gives
// every context an id that is never reused in the process, so a context
// destroyed and replaced (cudaDeviceReset, a caller's own cuCtxDestroy) can
// never be served a stale address.
struct ScratchEntry {
    unsigned long long ctx_id;
    void* address;
};
constexpr int kMaxScratchEntries = 64;
static std::mutex g_scratch_mutex;
static ScratchEntry g_scratch_entries[kMaxScratchEntries];
static int g_scratch_count = 0;

struct CtxFns {
    PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    PFN_cuCtxGetId_v12000 get_id = nullptr;
};

static const CtxFns& ctx_fns() {
    static CtxFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
        ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(ptr);
        cudaGetLastError();
    });
    return fns;
}

bool current_context_id(unsigned long long* id) {
    const CtxFns& f = ctx_fns();
    if (f.get_current == nullptr || f.get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return f.get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_noalloc_scratch in the current context.  In host code
// the array's name is only a host-side stand-in, so the real address must
// come from the runtime: cudaGetSymbolAddress, with the context current,
// checked, on the first call in each context.  It allocates nothing.
static pkv_status scratch_address(void** out) {
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    if (have_id) {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        for (int i = 0; i < g_scratch_count; ++i)
            if (g_scratch_entries[i].ctx_id == id) {
                *out = g_scratch_entries[i].address;
                return PKV_OK;
            }
    }
    // Set-up for this context.  (With no context current yet, this first
    // runtime call makes the device's primary context current.)
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    if (!have_id) have_id = current_context_id(&id);
    if (have_id) {
        std::lock_guard<std::mutex> lock(g_scratch_mutex);
        bool known = false;
        for (int i = 0; i < g_scratch_count; ++i) known |= g_scratch_entries[i].ctx_id == id;
        // more contexts than entries: later ones look the address up on every call
        if (!known && g_scratch_count < kMaxScratchEntries)
            g_scratch_entries[g_scratch_count++] = ScratchEntry{id, ptr};
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
    // The split plan of the 16-bit decode this call runs (the same plan
    // pkv_decode_attention makes for these arguments).
    size_t need = 0;
    if (decode_workspace_16bit(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                               max_context_len, num_splits, &need) != PKV_OK) {
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
