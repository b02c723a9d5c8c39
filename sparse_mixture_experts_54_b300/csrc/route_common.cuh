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
                                                int* hist = nullptr) {
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
    }
    if (logits_out && lane < n) logits_out[static_cast<size_t>(t) * n + lane] = mine;
}

}  // namespace moe
