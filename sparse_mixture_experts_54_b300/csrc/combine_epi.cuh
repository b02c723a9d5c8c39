// combine_epi.cuh -- the combine step of the layer fused into the W2 GEMM's
// epilogue.
//
// y[t] = sum over slots k of g_{t,k} * E_{idx[t][k]}(x_t) (aiqianji 2.1.1; the
// sum the code walkthrough does with index_add_, 3.1.2).  The W2 epilogue
// writes each gated expert row segment Ys[t*K + k][256 nb, 256 nb + 256) in
// fp32.  After writing one 128-feature block of such a row (and fencing it), a
// thread adds 1 to the counter of (token t, feature block); the thread that
// brings it to K is the last of the token's K rows there, and its warp adds
// the K rows in slot order (slot 0 first, then 1, ...) from L2, rounds once to
// bf16 (after adding the residual row h, when given) and writes y, then puts
// the counter back to 0 for the next call.  The
// sum and its order are the same whichever row arrives last, so y is bitwise
// reproducible.  Once the sum is written, the K slot-row segments are dead
// (nothing reads them again in this call, and the next call writes them before
// reading): the warp drops their L2 lines without writing them back to DRAM
// (discard.global.L2), so rows that are still in L2 never reach DRAM.
#pragma once

#include "common.cuh"

namespace moe {

struct CombineArgs {
    int* cnt;               // [T][d/128] arrival counters, zero between calls (null: no fused combine)
    __nv_bfloat16* y;       // [T][d]
    const __nv_bfloat16* resid;   // optional [T][d] added before the rounding (may be y itself)
    int K;
    int nblk;               // d / 128
    int d;
};

__device__ __forceinline__ float4 ldcg_f4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// Invalidate the 128-byte L2 line at p (128-byte aligned) without writing it back.
__device__ __forceinline__ void discard_l2_line(const void* p) {
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

// Called by all 32 lanes of an epilogue warp after each lane has written its
// row's features [128 blk, 128 blk + 128) of Ys (row = flat assignment a,
// valid or not; blk the same in every lane).
__device__ __forceinline__ void combine_arrive(const CombineArgs& c, const float* Ys, int ldY, bool valid, int a,
                                               int blk, int lane) {
    bool last = false;
    int t = 0;
    if (valid) {
        t = a / c.K;
        __threadfence();   // this row's Ys stores before the count
        last = atomicAdd(c.cnt + static_cast<size_t>(t) * c.nblk + blk, 1) == c.K - 1;
    }
    unsigned m = __ballot_sync(0xffffffffu, last);
    if (m == 0u) return;
    __threadfence();       // the count before the other rows' Ys loads
    __syncwarp();
    const int col = blk * 128 + 4 * lane;
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
        float4 s[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (r < nr) s[r] = ldcg_f4(Ys + static_cast<size_t>(tt[r]) * c.K * ldY + col);
        }
        for (int k = 1; k < c.K; ++k) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (r < nr) {
                    const float4 u = ldcg_f4(Ys + (static_cast<size_t>(tt[r]) * c.K + k) * ldY + col);
                    s[r].x += u.x; s[r].y += u.y; s[r].z += u.z; s[r].w += u.w;
                }
            }
        }
        if (c.resid) {
            // residual stream: y = h + (sum of the slot rows), one rounding
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if (r < nr) {
                    const uint2 hv = *reinterpret_cast<const uint2*>(c.resid + static_cast<size_t>(tt[r]) * c.d + col);
                    const __nv_bfloat162 h0 = *reinterpret_cast<const __nv_bfloat162*>(&hv.x);
                    const __nv_bfloat162 h1 = *reinterpret_cast<const __nv_bfloat162*>(&hv.y);
                    s[r].x = __low2float(h0) + s[r].x;
                    s[r].y = __high2float(h0) + s[r].y;
                    s[r].z = __low2float(h1) + s[r].z;
                    s[r].w = __high2float(h1) + s[r].w;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (r < nr) {
                uint2 o;
                o.x = pack_bf16x2(s[r].x, s[r].y);
                o.y = pack_bf16x2(s[r].z, s[r].w);
                *reinterpret_cast<uint2*>(c.y + static_cast<size_t>(tt[r]) * c.d + col) = o;
                if (lane == 0) c.cnt[static_cast<size_t>(tt[r]) * c.nblk + blk] = 0;
            }
        }
        // every lane's loads of the slot rows have been consumed above; lanes 0, 8,
        // 16 and 24 each drop one of the four 128-byte lines of a row's 512-byte segment
        __syncwarp();
        if ((lane & 7) == 0) {
            for (int r = 0; r < nr; ++r)
                for (int k = 0; k < c.K; ++k)
                    discard_l2_line(Ys + (static_cast<size_t>(tt[r]) * c.K + k) * ldY + blk * 128 + (lane >> 3) * 32);
        }
    }
}

}  // namespace moe
