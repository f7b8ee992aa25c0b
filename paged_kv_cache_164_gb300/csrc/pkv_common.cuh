// Device and host helpers shared by the pkv kernels (CUDA, sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// log2(e): scores are kept in base-2 units so the softmax uses exp2.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void flag_error(int32_t* err_flag, int bits) {
    if (err_flag != nullptr) atomicOr(err_flag, bits);
}

template <typename T> struct Pair;
template <> struct Pair<__half> { using type = __half2; };
template <> struct Pair<__nv_bfloat16> { using type = __nv_bfloat162; };

__device__ __forceinline__ float2 pair_to_float2(uint32_t bits, __half) {
    __half2 h = *reinterpret_cast<__half2*>(&bits);
    return __half22float2(h);
}
__device__ __forceinline__ float2 pair_to_float2(uint32_t bits, __nv_bfloat16) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&bits);
    return __bfloat1622float2(h);
}

__device__ __forceinline__ __half from_float(float x, __half) { return __float2half_rn(x); }
__device__ __forceinline__ __nv_bfloat16 from_float(float x, __nv_bfloat16) {
    return __float2bfloat16_rn(x);
}

// Loads N (2 or 4) consecutive 16-bit values as floats with one 4- or 8-byte load
// through the read-only path.
template <typename T, int N>
__device__ __forceinline__ void load_as_float(const T* ptr, float (&out)[N]) {
    static_assert(N == 2 || N == 4, "2 or 4 values per load");
    if constexpr (N == 2) {
        uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(ptr));
        float2 f = pair_to_float2(w, T());
        out[0] = f.x;
        out[1] = f.y;
    } else {
        uint2 w = __ldg(reinterpret_cast<const uint2*>(ptr));
        float2 a = pair_to_float2(w.x, T());
        float2 c = pair_to_float2(w.y, T());
        out[0] = a.x;
        out[1] = a.y;
        out[2] = c.x;
        out[3] = c.y;
    }
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool supported_head_dim(int d) { return d == 64 || d == 128; }
inline bool supported_block_size(int bs) { return bs == 16 || bs == 32 || bs == 64 || bs == 128; }

// The dtype argument of a call that takes the cache: the element type, with
// PKV_LAYOUT_HND OR-ed in for head-major caches.  Strips the flag and tells
// whether it was set.
inline bool take_layout(pkv_dtype& dtype) {
    const int v = static_cast<int>(dtype);
    dtype = static_cast<pkv_dtype>(v & ~PKV_LAYOUT_HND);
    return (v & PKV_LAYOUT_HND) != 0;
}

constexpr int kMaxGroup = 16;  // query heads per KV head served by one CTA

// Workspace bytes the 16-bit decode (pkv_decode_attention) plans for these
// arguments on the current device: the same plan decode_impl makes, not the
// larger of the 16-bit and E4M3 plans pkv_decode_workspace_size reports.
pkv_status decode_workspace_16bit(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int block_size, int max_context_len, int num_splits,
                                  size_t* bytes);

// Id of the CUDA context current to this thread (the one the launches use);
// false when none is current yet or the driver cannot say.  cuCtxGetId never
// reuses an id within a process, so per-context state keyed by it cannot be
// served to a context that replaced a destroyed one.
bool current_context_id(unsigned long long* id);

}  // namespace pkv
