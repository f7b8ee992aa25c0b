// Decode attention over a paged KV cache, split-K partitions and their
// log-sum-exp merge.
//
// The math: for one query token, s_t = scale * <q, K_t>, out = softmax(s) V
// (tutorial chapter 12, Attention(Q_t, K_1:t, V_1:t)), with the streaming
// online softmax m_new = max(m, s), l = e^(m - m_new) l + e^(s - m_new),
// O = e^(m - m_new) O + e^(s - m_new) V, one division at the end (vLLM deep
// dive 06, FlashAttention ③).  Long contexts are cut into KV partitions that
// run on different SMs and are merged with the same rescale rule
// (Flash-Decoding, ⑥; LLM-101-CN "推理优化" combine_result).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>

#include "pkv_common.cuh"

namespace pkv {

struct DecodeParams {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    float* partial_o;    // [B][H_q][num_splits][D] when num_splits > 1
    float* partial_lse;  // [B][H_q][num_splits]
    int32_t* err_flag;
    int max_blocks_per_seq;
    int num_blocks;
    int block_size;
    int num_q_heads;
    int num_kv_heads;
    int group;           // query heads per KV head
    int num_splits;
    int chunk_tokens;    // tokens per partition (a multiple of block_size)
    int max_context_len;
    float scale_log2;    // scale * log2(e)
};

constexpr int kDecodeWarps = 4;

// One CTA per (partition, KV head, sequence); its warps take the partition's
// pages round-robin and keep their own running (m, l, O) for every query head
// of the GQA group; the warps' states are combined at the end.  Lane j owns
// dimensions [j * D/32, (j + 1) * D/32).
template <typename T, int D, int GMAX>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_simple_kernel(DecodeParams p) {
    constexpr int VPT = D / 32;
    const int split = blockIdx.x;
    const int g = blockIdx.y;
    const int b = blockIdx.z;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int G = p.group;
    const int bs = p.block_size;

    int n = __ldg(p.context_lens + b);
    const int cap = min(p.max_blocks_per_seq * bs, p.max_context_len);
    if (n < 0 || n > cap) {
        if (split == 0 && threadIdx.x == 0) flag_error(p.err_flag, PKV_EFLAG_CONTEXT_LEN);
        n = n < 0 ? 0 : cap;
    }
    const int t_begin = split * p.chunk_tokens;
    const int t_end = min(n, t_begin + p.chunk_tokens);

    const T* q = static_cast<const T*>(p.q);
    float qf[GMAX][VPT];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
        if (h < G) {
            const T* qrow = q + ((int64_t)b * p.num_q_heads + g * G + h) * D + lane * VPT;
            load_as_float<T, VPT>(qrow, qf[h]);
#pragma unroll
            for (int i = 0; i < VPT; ++i) qf[h][i] *= p.scale_log2;
        } else {
#pragma unroll
            for (int i = 0; i < VPT; ++i) qf[h][i] = 0.f;
        }
    }

    float m[GMAX], l[GMAX], o[GMAX][VPT];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) o[h][i] = 0.f;
    }

    const T* kc = static_cast<const T*>(p.k_cache);
    const T* vc = static_cast<const T*>(p.v_cache);
    if (t_begin < t_end) {
        const int page_begin = t_begin / bs;
        const int page_end = (t_end + bs - 1) / bs;
        for (int pg = page_begin + warp; pg < page_end; pg += kDecodeWarps) {
            const int blk = __ldg(p.block_tables + (int64_t)b * p.max_blocks_per_seq + pg);
            if (blk < 0 || blk >= p.num_blocks) {
                if (lane == 0) flag_error(p.err_flag, PKV_EFLAG_BLOCK_ID);
                continue;
            }
            const int tb = max(pg * bs, t_begin);
            const int te = min(pg * bs + bs, t_end);
            for (int t = tb; t < te; ++t) {
                const int64_t row =
                    (((int64_t)blk * bs + (t - pg * bs)) * p.num_kv_heads + g) * D + lane * VPT;
                float kf[VPT], vf[VPT];
                load_as_float<T, VPT>(kc + row, kf);
                load_as_float<T, VPT>(vc + row, vf);
#pragma unroll
                for (int h = 0; h < GMAX; ++h) {
                    if (h >= G) break;
                    float s = 0.f;
#pragma unroll
                    for (int i = 0; i < VPT; ++i) s = fmaf(qf[h][i], kf[i], s);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
                    const float m_new = fmaxf(m[h], s);
                    const float alpha = exp2f(m[h] - m_new);  // 0 when m was -inf
                    const float e = exp2f(s - m_new);
                    l[h] = l[h] * alpha + e;
#pragma unroll
                    for (int i = 0; i < VPT; ++i) o[h][i] = fmaf(o[h][i], alpha, e * vf[i]);
                    m[h] = m_new;
                }
            }
        }
    }

    // Combine the warps' (m, l, O) per query head.
    __shared__ float sm_m[kDecodeWarps][GMAX];
    __shared__ float sm_l[kDecodeWarps][GMAX];
    __shared__ float sm_o[kDecodeWarps][GMAX][D];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
        if (lane == 0) {
            sm_m[warp][h] = m[h];
            sm_l[warp][h] = l[h];
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) sm_o[warp][h][lane * VPT + i] = o[h][i];
    }
    __syncthreads();

    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int h = idx / D;
        const int j = idx % D;
        float mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kDecodeWarps; ++w) mx = fmaxf(mx, sm_m[w][h]);
        float acc = 0.f, den = 0.f;
        if (mx != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kDecodeWarps; ++w) {
                const float mw = sm_m[w][h];
                if (mw == -INFINITY) continue;
                const float c = exp2f(mw - mx);
                den = fmaf(sm_l[w][h], c, den);
                acc = fmaf(sm_o[w][h][j], c, acc);
            }
        }
        const float val = den > 0.f ? acc / den : 0.f;
        const int hq = g * G + h;
        if (p.num_splits == 1) {
            T* out = static_cast<T*>(p.out);
            out[((int64_t)b * p.num_q_heads + hq) * D + j] = from_float(val, T());
        } else {
            const int64_t row = ((int64_t)b * p.num_q_heads + hq) * p.num_splits + split;
            p.partial_o[row * D + j] = val;
            if (j == 0) p.partial_lse[row] = den > 0.f ? (mx + log2f(den)) * kLn2 : -INFINITY;
        }
    }
}

// Merge: one CTA per (sequence, query head); thread j produces dimension j.
template <typename T>
__global__ void __launch_bounds__(128)
merge_kernel(T* __restrict__ out, const float* __restrict__ partial_o,
             const float* __restrict__ partial_lse, int num_splits, int head_dim) {
    const int64_t row = blockIdx.x;  // b * H_q + h
    const float* lse = partial_lse + row * num_splits;
    float mx = -INFINITY;
    for (int s = 0; s < num_splits; ++s) mx = fmaxf(mx, __ldg(lse + s));
    for (int j = threadIdx.x; j < head_dim; j += blockDim.x) {
        float acc = 0.f, den = 0.f;
        if (mx != -INFINITY) {
            for (int s = 0; s < num_splits; ++s) {
                const float ls = __ldg(lse + s);
                if (ls == -INFINITY) continue;
                const float w = expf(ls - mx);
                den += w;
                acc = fmaf(w, __ldg(partial_o + (row * num_splits + s) * head_dim + j), acc);
            }
        }
        out[row * head_dim + j] = from_float(den > 0.f ? acc / den : 0.f, T());
    }
}

// ---------------------------------------------------------------------------
// Host side: split planning, dispatch
// ---------------------------------------------------------------------------

static int current_sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (dev < 0 || dev >= 64) return -1;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return -1;
    }
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

struct Plan {
    int num_splits;
    int chunk_tokens;
    size_t workspace_bytes;
};

// Validates the shape arguments shared by planning and launching.
static pkv_status check_shapes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, int max_context_len, int num_splits) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0 || max_context_len < 0 || num_splits < 0 || num_splits > PKV_MAX_SPLITS)
        return PKV_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim) || !supported_block_size(block_size) ||
        num_q_heads / num_kv_heads > kMaxGroup)
        return PKV_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

static pkv_status make_plan(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_context_len, int num_splits, Plan* plan) {
    pkv_status st = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_context_len, num_splits);
    if (st != PKV_OK) return st;
    const int max_pages = max(1, (max_context_len + block_size - 1) / block_size);
    int splits = num_splits;
    if (splits == 0) {
        const int sms = current_sm_count();
        if (sms <= 0) return PKV_ERR_CUDA;
        const int64_t units = (int64_t)max(1, num_seqs) * num_kv_heads;
        const int64_t target = 4LL * sms;
        splits = (int)std::min<int64_t>(PKV_MAX_SPLITS, (target + units - 1) / units);
        // keep at least 8 pages per partition
        splits = min(splits, max(1, max_pages / 8));
    }
    splits = max(1, min(splits, max_pages));
    const int chunk_pages = (max_pages + splits - 1) / splits;
    splits = (max_pages + chunk_pages - 1) / chunk_pages;
    plan->num_splits = splits;
    plan->chunk_tokens = chunk_pages * block_size;
    plan->workspace_bytes =
        splits > 1 ? (size_t)num_seqs * num_q_heads * splits * (head_dim + 1) * sizeof(float) + 256
                   : 0;
    return PKV_OK;
}

template <typename T, int D>
static void launch_decode_d(const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    const int G = p.group;
    if (G == 1)
        decode_simple_kernel<T, D, 1><<<grid, kDecodeWarps * 32, 0, stream>>>(p);
    else if (G == 2)
        decode_simple_kernel<T, D, 2><<<grid, kDecodeWarps * 32, 0, stream>>>(p);
    else if (G <= 4)
        decode_simple_kernel<T, D, 4><<<grid, kDecodeWarps * 32, 0, stream>>>(p);
    else if (G <= 8)
        decode_simple_kernel<T, D, 8><<<grid, kDecodeWarps * 32, 0, stream>>>(p);
    else
        decode_simple_kernel<T, D, 16><<<grid, kDecodeWarps * 32, 0, stream>>>(p);
}

template <typename T>
static void launch_decode(const DecodeParams& p, int head_dim, dim3 grid, cudaStream_t stream) {
    if (head_dim == 64)
        launch_decode_d<T, 64>(p, grid, stream);
    else
        launch_decode_d<T, 128>(p, grid, stream);
}

}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_dim, int block_size, int max_context_len,
                                            int num_splits) {
    Plan plan;
    if (make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                  num_splits, &plan) != PKV_OK)
        return SIZE_MAX;
    return plan.workspace_bytes;
}

extern "C" int pkv_decode_num_splits(int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int max_context_len,
                                     int num_splits) {
    Plan plan;
    if (make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                  num_splits, &plan) != PKV_OK)
        return -1;
    return plan.num_splits;
}

extern "C" pkv_status pkv_decode_attention(void* out, const void* q, const void* k_cache,
                                           const void* v_cache, const int32_t* block_tables,
                                           int max_blocks_per_seq, const int32_t* context_lens,
                                           int max_context_len, int num_seqs, int num_blocks,
                                           int block_size, int num_q_heads, int num_kv_heads,
                                           int head_dim, float scale, int num_splits,
                                           void* workspace, size_t workspace_bytes,
                                           pkv_dtype dtype, int32_t* err_flag, void* stream) {
    pkv_status st = check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_context_len, num_splits);
    if (st != PKV_OK) return st;
    if ((dtype != PKV_FP16 && dtype != PKV_BF16) || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
        !std::isfinite(scale))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PKV_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
        (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PKV_ERR_INVALID_ARG;
    Plan plan;
    st = make_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_context_len,
                   num_splits, &plan);
    if (st != PKV_OK) return st;
    if (plan.workspace_bytes > 0 && (workspace == nullptr || workspace_bytes < plan.workspace_bytes))
        return PKV_ERR_WORKSPACE;
    if (workspace != nullptr && !aligned16(workspace)) return PKV_ERR_INVALID_ARG;

    DecodeParams p;
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.err_flag = err_flag;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_q_heads / num_kv_heads;
    p.num_splits = plan.num_splits;
    p.chunk_tokens = plan.chunk_tokens;
    p.max_context_len = max_context_len;
    p.scale_log2 = scale * kLog2e;
    p.partial_o = nullptr;
    p.partial_lse = nullptr;
    if (plan.num_splits > 1) {
        p.partial_o = static_cast<float*>(workspace);
        p.partial_lse = p.partial_o + (size_t)num_seqs * num_q_heads * plan.num_splits * head_dim;
    }
    cudaStream_t s = (cudaStream_t)stream;
    dim3 grid(plan.num_splits, num_kv_heads, num_seqs);
    if (dtype == PKV_FP16)
        launch_decode<__half>(p, head_dim, grid, s);
    else
        launch_decode<__nv_bfloat16>(p, head_dim, grid, s);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    if (plan.num_splits > 1) {
        const int rows = num_seqs * num_q_heads;
        if (dtype == PKV_FP16)
            merge_kernel<__half><<<rows, 128, 0, s>>>(static_cast<__half*>(out), p.partial_o,
                                                      p.partial_lse, plan.num_splits, head_dim);
        else
            merge_kernel<__nv_bfloat16><<<rows, 128, 0, s>>>(static_cast<__nv_bfloat16*>(out),
                                                             p.partial_o, p.partial_lse,
                                                             plan.num_splits, head_dim);
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    }
    return PKV_OK;
}

extern "C" pkv_status pkv_merge(void* out, const float* partial_o, const float* partial_lse,
                                int num_seqs, int num_q_heads, int num_splits, int head_dim,
                                pkv_dtype dtype, void* stream) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_splits <= 0 || head_dim <= 0 ||
        (dtype != PKV_FP16 && dtype != PKV_BF16))
        return PKV_ERR_INVALID_ARG;
    if (num_seqs == 0) return PKV_OK;
    if (!out || !partial_o || !partial_lse) return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(out) & 1u) || (reinterpret_cast<uintptr_t>(partial_o) & 3u) ||
        (reinterpret_cast<uintptr_t>(partial_lse) & 3u))
        return PKV_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)num_seqs * num_q_heads;
    if (rows > INT_MAX) return PKV_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    if (dtype == PKV_FP16)
        merge_kernel<__half><<<(int)rows, 128, 0, s>>>(static_cast<__half*>(out), partial_o,
                                                       partial_lse, num_splits, head_dim);
    else
        merge_kernel<__nv_bfloat16><<<(int)rows, 128, 0, s>>>(
            static_cast<__nv_bfloat16*>(out), partial_o, partial_lse, num_splits, head_dim);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
