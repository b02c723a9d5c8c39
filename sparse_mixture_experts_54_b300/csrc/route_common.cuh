// route_common.cuh -- per-token pieces of the router shared by the routing
// kernels: fp32 loads of a row, and the top-k selection + gate of one token.
//
// G(x) = Softmax(TopK(x . W_g)): the K largest logits are kept, the rest count
// as -inf (Mixtral of Experts section 2.1, restated in aiqianji 2.1.1).
#pragma once

#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------------------
// 8 consecutive elements of a row as fp32 (zeros past the end of the row).
template <typename TX>
__device__ __forceinline__ void load8(const TX* row, int j0, int d, float (&v)[8]) {
    if (j0 >= d) {
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = 0.0f;
        return;
    }
    if constexpr (sizeof(TX) == 2) {
        uint4 raw = __ldg(reinterpret_cast<const uint4*>(row + j0));
        const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = __bfloat162float(h[u]);
    } else {
        float4 a = __ldg(reinterpret_cast<const float4*>(row + j0));
        float4 b = __ldg(reinterpret_cast<const float4*>(row + j0 + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// Top-k and gate from the n logits held (identically) by every lane of a warp:
// lane e ranks its own expert (number of experts with a larger logit, or an
// equal logit at a lower index); the K best write their slot.  Softmax over
// the kept logits only (the others are -inf), shifted by the maximum.
template <int NMAX>
__device__ __forceinline__ void topk_gate_write(const float (&l)[NMAX], int n, int K, int t, int lane,
                                                int32_t* topk_idx, float* topk_w, float* logits_out,
                                                int* hist = nullptr, int* local_idx = nullptr) {
    float mine = 0.0f, lmax = -INFINITY;
#pragma unroll
    for (int e = 0; e < NMAX; ++e) {
        if (e < n) {
            if (e == lane) mine = l[e];
            lmax = fmaxf(lmax, l[e]);
        }
    }
    int rank = 0;
#pragma unroll
    for (int e = 0; e < NMAX; ++e) {
        if (e < n) rank += (l[e] > mine) || (l[e] == mine && e < lane);
    }
    const bool kept = lane < n && rank < K;
    const float num = kept ? expf(mine - lmax) : 0.0f;
    float z = num;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    if (kept) {
        topk_idx[static_cast<size_t>(t) * K + rank] = lane;
        topk_w[static_cast<size_t>(t) * K + rank] = num / z;
        if (hist) atomicAdd(hist + lane, 1);   // a count: the order of the adds does not matter
        if (local_idx) local_idx[rank] = lane;  // the same choice, for a caller that reads it back soon
    }
    if (logits_out && lane < n) logits_out[static_cast<size_t>(t) * n + lane] = mine;
}

// ---------------------------------------------------------------------------
// Global-memory flag words of the grid-wide barriers.
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Pieces of the router's per-token arithmetic (route_fused.cu), shared by every
// kernel that routes, so that they all take the same fp32 decisions.

// x * s rounded to the element type (bf16: round to nearest even; fp32: as is).
template <typename TX>
__device__ __forceinline__ float scale_round(float x, float s) {
    if constexpr (sizeof(TX) == 2) return __bfloat162float(__float2bfloat16_rn(x * s));
    return x * s;
}

// Sum over the 32 lanes of V values per lane (V a power of two).  Each step
// trades half of the values with the partner lane and adds, halving the count,
// until one value per lane is left; remaining steps are plain butterflies.
// Afterwards lane l holds the full sums of value indices fr_index(l, i),
// i < max(V/32, 1).
template <int V>
__device__ __forceinline__ void lane_transpose_sum(float (&v)[V], int lane) {
    int cur = V;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        if (cur > 1) {
            const int half = cur >> 1;
            const bool up = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < V / 2; ++i) {
                if (i < half) {
                    const float send = up ? v[i] : v[half + i];
                    const float keep = up ? v[half + i] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            cur = half;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
}
// 4 consecutive elements of a row as loaded (bf16: 8 bytes, fp32: 16 bytes),
// so that the next segment's loads can be in flight while one is computed.
template <typename TX>
struct Raw4;
template <>
struct Raw4<__nv_bfloat16> {
    uint2 v;
};
template <>
struct Raw4<float> {
    float4 v;
};
template <typename TX>
__device__ __forceinline__ void load_raw4(const TX* row, int j0, bool ok, Raw4<TX>& r) {
    if constexpr (sizeof(TX) == 2) {
        r.v = ok ? __ldg(reinterpret_cast<const uint2*>(row + j0)) : make_uint2(0u, 0u);
    } else {
        r.v = ok ? __ldg(reinterpret_cast<const float4*>(row + j0)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
template <typename TX>
__device__ __forceinline__ void unpack_raw4(const Raw4<TX>& r, float* v) {
    if constexpr (sizeof(TX) == 2) {
        const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&r.v.x);
        const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&r.v.y);
        v[0] = __low2float(lo);
        v[1] = __high2float(lo);
        v[2] = __low2float(hi);
        v[3] = __high2float(hi);
    } else {
        v[0] = r.v.x; v[1] = r.v.y; v[2] = r.v.z; v[3] = r.v.w;
    }
}

// 16 bytes of a row (8 bf16 or 4 fp32), each element times s, rounded back.
template <typename TX>
__device__ __forceinline__ uint4 scale_row_vec(uint4 v, float s) {
    if constexpr (sizeof(TX) == 2) {
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
            const __nv_bfloat162 o = __floats2bfloat162_rn(__low2float(b) * s, __high2float(b) * s);
            w[i] = *reinterpret_cast<const uint32_t*>(&o);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        return make_uint4(__float_as_uint(__uint_as_float(v.x) * s), __float_as_uint(__uint_as_float(v.y) * s),
                          __float_as_uint(__uint_as_float(v.z) * s), __float_as_uint(__uint_as_float(v.w) * s));
    }
}

template <int V>
__device__ __forceinline__ int fr_index(int lane, int i) {
    int idx = i, cur = V;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        if (cur > 1) {
            cur >>= 1;
            if (lane & o) idx += cur;
        }
    }
    return idx;
}

}  // namespace moe
