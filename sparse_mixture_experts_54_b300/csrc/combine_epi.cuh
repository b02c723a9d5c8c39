// combine_epi.cuh -- the combine step of the layer fused into the W2 GEMM's
// epilogue.
//
// y[t] = sum over slots k of g_{t,k} * E_{idx[t][k]}(x_t) (aiqianji 2.1.1; the
// sum the code walkthrough does with index_add_, 3.1.2).  The W2 epilogue
// writes each gated expert row segment Ys[t*K + k][256 nb, 256 nb + 256) in
// fp32.  After writing one (and fencing it), a thread adds 1 to the counter of
// (token t, feature block nb); the thread that brings it to K is the last of
// the token's K rows there, and its warp adds the K rows in slot order
// (slot 0 first, then 1, ...) from L2, rounds once to bf16 and writes y, then
// puts the counter back to 0 for the next call.  The sum and its order are the
// same whichever row arrives last, so y is bitwise reproducible.
#pragma once

#include "common.cuh"

namespace moe {

struct CombineArgs {
    int* cnt;               // [T][d/256] arrival counters, zero between calls (null: no fused combine)
    __nv_bfloat16* y;       // [T][d]
    int K;
    int nblk;               // d / 256
    int d;
};

__device__ __forceinline__ float4 ldcg_f4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// Called by all 32 lanes of an epilogue warp after each lane has written its
// row's 256-feature segment of Ys (row = flat assignment a, valid or not).
__device__ __forceinline__ void combine_arrive(const CombineArgs& c, const float* Ys, int ldY, bool valid, int a,
                                               int nb, int lane) {
    bool last = false;
    int t = 0;
    if (valid) {
        t = a / c.K;
        __threadfence();   // this row's Ys stores before the count
        last = atomicAdd(c.cnt + static_cast<size_t>(t) * c.nblk + nb, 1) == c.K - 1;
    }
    unsigned m = __ballot_sync(0xffffffffu, last);
    if (m == 0u) return;
    __threadfence();       // the count before the other rows' Ys loads
    __syncwarp();
    const int col = nb * 256 + 8 * lane;
    while (m) {
        int tt[4];
        int nr = 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            tt[r] = 0;
            if (m) {
                const int src = __ffs(m) - 1;
                m &= m - 1;
                tt[r] = src;
                ++nr;
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) tt[r] = __shfl_sync(0xffffffffu, t, tt[r]);
        float4 s[4][2];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (r < nr) {
                const float* row = Ys + static_cast<size_t>(tt[r]) * c.K * ldY + col;
                s[r][0] = ldcg_f4(row);
                s[r][1] = ldcg_f4(row + 4);
            }
        }
        for (int k = 1; k < c.K; ++k) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (r < nr) {
                    const float* row = Ys + (static_cast<size_t>(tt[r]) * c.K + k) * ldY + col;
                    const float4 u0 = ldcg_f4(row), u1 = ldcg_f4(row + 4);
                    s[r][0].x += u0.x; s[r][0].y += u0.y; s[r][0].z += u0.z; s[r][0].w += u0.w;
                    s[r][1].x += u1.x; s[r][1].y += u1.y; s[r][1].z += u1.z; s[r][1].w += u1.w;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (r < nr) {
                uint4 o;
                o.x = pack_bf16x2(s[r][0].x, s[r][0].y);
                o.y = pack_bf16x2(s[r][0].z, s[r][0].w);
                o.z = pack_bf16x2(s[r][1].x, s[r][1].y);
                o.w = pack_bf16x2(s[r][1].z, s[r][1].w);
                *reinterpret_cast<uint4*>(c.y + static_cast<size_t>(tt[r]) * c.d + col) = o;
                if (lane == 0) c.cnt[static_cast<size_t>(tt[r]) * c.nblk + nb] = 0;
            }
        }
    }
}

}  // namespace moe
