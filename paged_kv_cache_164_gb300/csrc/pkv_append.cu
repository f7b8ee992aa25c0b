// Append (scatter through slot_mapping) and block-table gather, plus the
// status helpers of the C ABI.
//
// Append: token i with slot s >= 0 is written to block s / block_size at offset
// s % block_size (gsyq.cn essay §三.2 get_kv_cache; tutorial chapter 12
// PagedKVCache.update; LLM-101-CN "推理优化" KVCachePool.write_tokens).
// One CTA per token; the token's K and V rows ([num_kv_heads][head_dim], a
// multiple of 16 bytes) are moved with 16-byte vector loads and stores.  In a
// head-major cache ([num_blocks][num_kv_heads][block_size][head_dim]) head g
// of the token lands in the (block, g) tile at row offset.
#include <climits>
#include <cmath>

#include <cuda_fp8.h>

#include "pkv_common.cuh"

namespace pkv {

// Offset (in 16-byte vectors) of vector c of a token's [num_kv_heads][head_dim]
// row at `slot` of the cache.
__device__ __forceinline__ int64_t cache_vec(int64_t slot, int c, int row_vecs, int head_vecs,
                                             int num_kv_heads, int block_size, bool hnd) {
    if (!hnd) return slot * row_vecs + c;
    const int64_t blk = slot / block_size;
    const int off = (int)(slot - blk * block_size);
    const int g = c / head_vecs;
    return ((blk * num_kv_heads + g) * block_size + off) * head_vecs + (c - g * head_vecs);
}

__global__ void __launch_bounds__(128)
append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
              uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
              const int64_t* __restrict__ slot_mapping, int64_t num_slots, int row_vecs,
              int head_vecs, int num_kv_heads, int block_size, bool hnd, int32_t* err_flag) {
    // Launched as a programmatic dependent: let the next kernel (the decode)
    // get scheduled now, then wait for the previous one before touching memory.
    asm volatile("griddepcontrol.launch_dependents;" :::);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int i = blockIdx.x;
    const int64_t slot = __ldg(slot_mapping + i);
    if (slot < 0) return;  // padding
    if (slot >= num_slots) {
        if (threadIdx.x == 0) flag_error(err_flag, PKV_EFLAG_SLOT);
        return;
    }
    // Token-major: [num_blocks][block_size] flattens to the slot index itself.
    const uint4* ks = k_new + (int64_t)i * row_vecs;
    const uint4* vs = v_new + (int64_t)i * row_vecs;
    for (int c = threadIdx.x; c < row_vecs; c += blockDim.x) {
        const int64_t d = cache_vec(slot, c, row_vecs, head_vecs, num_kv_heads, block_size, hnd);
        uint4 a = __ldg(ks + c);
        uint4 b = __ldg(vs + c);
        k_cache[d] = a;
        v_cache[d] = b;
    }
}

// Gather: one CTA per (page of the block table, sequence).  Tokens of the page
// below the sequence's context are copied row by row into the contiguous output.
__global__ void __launch_bounds__(128)
gather_kernel(uint4* __restrict__ k_out, uint4* __restrict__ v_out,
              const uint4* __restrict__ k_cache, const uint4* __restrict__ v_cache,
              const int32_t* __restrict__ block_tables, int max_blocks_per_seq,
              const int32_t* __restrict__ context_lens, int max_context_len, int num_blocks,
              int block_size, int row_vecs, int head_vecs, int num_kv_heads, bool hnd,
              int32_t* err_flag) {
    const int page = blockIdx.x;
    const int b = blockIdx.y;
    int n = __ldg(context_lens + b);
    const int cap = min(max_blocks_per_seq * block_size, max_context_len);
    if (n < 0 || n > cap) {
        if (page == 0 && threadIdx.x == 0) flag_error(err_flag, PKV_EFLAG_CONTEXT_LEN);
        n = n < 0 ? 0 : cap;
    }
    const int t0 = page * block_size;
    if (t0 >= n) return;
    const int t1 = min(n, t0 + block_size);
    const int blk = __ldg(block_tables + (int64_t)b * max_blocks_per_seq + page);
    if (blk < 0 || blk >= num_blocks) {
        if (threadIdx.x == 0) flag_error(err_flag, PKV_EFLAG_BLOCK_ID);
        return;
    }
    const int total = (t1 - t0) * row_vecs;
    for (int c = threadIdx.x; c < total; c += blockDim.x) {
        const int t = t0 + c / row_vecs;
        const int v = c % row_vecs;
        const int64_t src = cache_vec((int64_t)blk * block_size + (t - t0), v, row_vecs,
                                      head_vecs, num_kv_heads, block_size, hnd);
        const int64_t dst = ((int64_t)b * max_context_len + t) * row_vecs + v;
        k_out[dst] = __ldg(k_cache + src);
        v_out[dst] = __ldg(v_cache + src);
    }
}

// Quantising append into an E4M3 cache (vLLM deep dive, 3.3 FP8 inference:
// E4M3 with the range held by a scale; 2.2: the KV-cache write fused with
// quantisation): element x of token i's K row is stored as E4M3(x / k_scale),
// the quotient rounded to fp32 and then to the nearest E4M3 value (ties to
// even), saturating at +-448; likewise V.  One CTA per token, eight elements
// (16 input bytes, 8 output bytes) per thread and step.
template <typename T>
__global__ void __launch_bounds__(128)
append_fp8_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                  uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                  const int64_t* __restrict__ slot_mapping, int64_t num_slots, int num_kv_heads,
                  int head_dim, int block_size, bool hnd, float k_scale, float v_scale,
                  int32_t* err_flag) {
    asm volatile("griddepcontrol.launch_dependents;" :::);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int i = blockIdx.x;
    const int64_t slot = __ldg(slot_mapping + i);
    if (slot < 0) return;  // padding
    if (slot >= num_slots) {
        if (threadIdx.x == 0) flag_error(err_flag, PKV_EFLAG_SLOT);
        return;
    }
    const int row = num_kv_heads * head_dim;
    const int64_t blk = slot / block_size;
    const int off = (int)(slot - blk * block_size);
    for (int c = threadIdx.x; c < row / 8; c += blockDim.x) {
        const int e = c * 8;              // element of the [heads][dim] row
        const int g = e / head_dim;
        const int64_t dst = hnd ? ((blk * num_kv_heads + g) * block_size + off) * head_dim +
                                      (e - g * head_dim)
                                : slot * row + e;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint4 raw = __ldg((which ? v_new : k_new) + ((int64_t)i * row + e) / 8);
            const float sc = which ? v_scale : k_scale;
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t outw[2] = {0u, 0u};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 x = pair_to_float2(w[j], T());
                const float2 f = make_float2(__fdiv_rn(x.x, sc), __fdiv_rn(x.y, sc));
                const uint32_t two = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3);
                outw[j / 2] |= two << (16 * (j % 2));
            }
            *reinterpret_cast<uint2*>((which ? v_cache : k_cache) + dst) =
                make_uint2(outw[0], outw[1]);
        }
    }
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_append(const void* k_new, const void* v_new, void* k_cache,
                                 void* v_cache, const int64_t* slot_mapping, int num_tokens,
                                 int num_blocks, int block_size, int num_kv_heads, int head_dim,
                                 pkv_dtype dtype, int32_t* err_flag, void* stream) {
    const bool hnd = take_layout(dtype);
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || (dtype != PKV_FP16 && dtype != PKV_BF16))
        return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PKV_ERR_INVALID_ARG;
    const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * 2;
    if (row_bytes % 16 != 0 || row_bytes / 16 > INT_MAX) return PKV_ERR_UNSUPPORTED;
    if (hnd && (head_dim * 2) % 16 != 0) return PKV_ERR_UNSUPPORTED;
    const int row_vecs = (int)(row_bytes / 16);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_tokens);
    cfg.blockDim = dim3(128);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, append_kernel, (const uint4*)k_new, (const uint4*)v_new, (uint4*)k_cache,
        (uint4*)v_cache, slot_mapping, (int64_t)num_blocks * block_size, row_vecs, head_dim / 8,
        num_kv_heads, block_size, hnd, err_flag);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" pkv_status pkv_gather(void* k_out, void* v_out, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 int max_blocks_per_seq, const int32_t* context_lens,
                                 int max_context_len, int num_seqs, int num_blocks,
                                 int block_size, int num_kv_heads, int head_dim, pkv_dtype dtype,
                                 int32_t* err_flag, void* stream) {
    const bool hnd = take_layout(dtype);
    if (num_seqs < 0 || max_context_len < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        (dtype != PKV_FP16 && dtype != PKV_BF16))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0 || max_context_len == 0) return PKV_OK;
    if (!k_out || !v_out || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_out) || !aligned16(v_out) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PKV_ERR_INVALID_ARG;
    const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * 2;
    if (row_bytes % 16 != 0 || row_bytes / 16 > INT_MAX) return PKV_ERR_UNSUPPORTED;
    if (hnd && (head_dim * 2) % 16 != 0) return PKV_ERR_UNSUPPORTED;
    const int pages = (max_context_len + block_size - 1) / block_size;
    if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
    dim3 grid(pages, num_seqs);
    gather_kernel<<<grid, 128, 0, (cudaStream_t)stream>>>(
        (uint4*)k_out, (uint4*)v_out, (const uint4*)k_cache, (const uint4*)v_cache, block_tables,
        max_blocks_per_seq, context_lens, max_context_len, num_blocks, block_size,
        (int)(row_bytes / 16), head_dim / 8, num_kv_heads, hnd, err_flag);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" pkv_status pkv_check_error(const int32_t* err_flag, void* stream,
                                      int32_t* flags_out) {
    if (err_flag == nullptr) return PKV_ERR_INVALID_ARG;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return PKV_ERR_CUDA;
    int32_t word = 0;
    if (cudaMemcpy(&word, err_flag, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (flags_out) *flags_out = word;
    if (word == 0) return PKV_OK;
    if (word & PKV_EFLAG_TIMEOUT) return PKV_ERR_DEVICE_TIMEOUT;
    return PKV_ERR_DEVICE_INDEX;
}

extern "C" const char* pkv_status_string(pkv_status status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported size or type";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_CUDA: return "CUDA runtime error";
        case PKV_ERR_DEVICE_INDEX: return "a kernel skipped an out-of-range index";
        case PKV_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel expired";
    }
    return "unknown status";
}

extern "C" int pkv_max_group_size(void) { return kMaxGroup; }

extern "C" int pkv_debug_build(void) {
#ifdef PKV_DEBUG
    return 1;
#else
    return 0;
#endif
}

extern "C" pkv_status pkv_append_fp8(const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, const int64_t* slot_mapping, int num_tokens,
                                     int num_blocks, int block_size, int num_kv_heads,
                                     int head_dim, float k_scale, float v_scale, pkv_dtype dtype,
                                     int32_t* err_flag, void* stream) {
    const bool hnd = take_layout(dtype);
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || (dtype != PKV_FP16 && dtype != PKV_BF16) || !std::isfinite(k_scale) ||
        !std::isfinite(v_scale) || k_scale <= 0.f || v_scale <= 0.f)
        return PKV_ERR_INVALID_ARG;
    if (head_dim % 8 != 0) return PKV_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(k_cache) & 7u) ||
        (reinterpret_cast<uintptr_t>(v_cache) & 7u) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)num_kv_heads * head_dim > INT_MAX / 2) return PKV_ERR_UNSUPPORTED;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_tokens);
    cfg.blockDim = dim3(128);
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int64_t slots = (int64_t)num_blocks * block_size;
    const cudaError_t e =
        dtype == PKV_FP16
            ? cudaLaunchKernelEx(&cfg, append_fp8_kernel<__half>, (const uint4*)k_new,
                                 (const uint4*)v_new, (uint8_t*)k_cache, (uint8_t*)v_cache,
                                 slot_mapping, slots, num_kv_heads, head_dim, block_size, hnd,
                                 k_scale, v_scale, err_flag)
            : cudaLaunchKernelEx(&cfg, append_fp8_kernel<__nv_bfloat16>, (const uint4*)k_new,
                                 (const uint4*)v_new, (uint8_t*)k_cache, (uint8_t*)v_cache,
                                 slot_mapping, slots, num_kv_heads, head_dim, block_size, hnd,
                                 k_scale, v_scale, err_flag);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_CUDA;
    }
    return PKV_OK;
}
