// route.cu -- router logits + top-k gate, deterministic dispatch, row gather,
// and the fixed-order combine of each token's expert rows.
//
// Router: G(x) = Softmax(TopK(x . W_g)), TopK keeping the K largest logits
// (Mixtral of Experts section 2.1, restated in aiqianji section 2.1.1; router
// is nn.Linear(hidden_dim, num_experts, bias=False), aiqianji 2.1.4).
// Dispatch replaces the one_hot/permute/where walk and the row gather of
// aiqianji 3.1.2 (code blocks B, C); combine replaces index_add_ there.
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------------------
// Router: one warp per token.  W_g [n][d] fp32 is staged once per block in
// shared memory; each lane owns 8 consecutive elements of every 256-element
// slice of the row, sums its partial dot products in a fixed order and the
// warp adds the lanes with a butterfly, so every lane holds all n logits and
// the result does not depend on timing.
template <typename TX, int NMAX>
__global__ void __launch_bounds__(512) router_topk_kernel(const TX* __restrict__ x,
                                                          const float* __restrict__ Wg,
                                                          const float* __restrict__ bias, int T,
                                                          int d, int n, int K,
                                                          int32_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_w,
                                                          float* __restrict__ logits_out) {
    extern __shared__ float wg_s[];
    for (int i = threadIdx.x * 4; i < n * d; i += blockDim.x * 4)
        *reinterpret_cast<float4*>(wg_s + i) = __ldg(reinterpret_cast<const float4*>(Wg + i));
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    for (int t = blockIdx.x * warps + (threadIdx.x >> 5); t < T; t += gridDim.x * warps) {
        float acc[NMAX];
#pragma unroll
        for (int e = 0; e < NMAX; ++e) acc[e] = 0.0f;
        const TX* xr = x + static_cast<size_t>(t) * d;
        for (int j0 = lane * 8; j0 < d; j0 += 256) {
            float xv[8];
            if constexpr (sizeof(TX) == 2) {
                uint4 raw = __ldg(reinterpret_cast<const uint4*>(xr + j0));
                const __nv_bfloat16* h = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
                for (int u = 0; u < 8; ++u) xv[u] = __bfloat162float(h[u]);
            } else {
                float4 a = __ldg(reinterpret_cast<const float4*>(xr + j0));
                float4 b = __ldg(reinterpret_cast<const float4*>(xr + j0 + 4));
                xv[0] = a.x; xv[1] = a.y; xv[2] = a.z; xv[3] = a.w;
                xv[4] = b.x; xv[5] = b.y; xv[6] = b.z; xv[7] = b.w;
            }
#pragma unroll
            for (int e = 0; e < NMAX; ++e) {
                if (e < n) {
                    const float* w = wg_s + e * d + j0;
                    float4 w0 = *reinterpret_cast<const float4*>(w);
                    float4 w1 = *reinterpret_cast<const float4*>(w + 4);
                    float a = acc[e];
                    a = fmaf(xv[0], w0.x, a); a = fmaf(xv[1], w0.y, a);
                    a = fmaf(xv[2], w0.z, a); a = fmaf(xv[3], w0.w, a);
                    a = fmaf(xv[4], w1.x, a); a = fmaf(xv[5], w1.y, a);
                    a = fmaf(xv[6], w1.z, a); a = fmaf(xv[7], w1.w, a);
                    acc[e] = a;
                }
            }
        }
        // butterfly sum: identical result in every lane
#pragma unroll
        for (int e = 0; e < NMAX; ++e) {
            if (e < n) {
                float v = acc[e];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                acc[e] = v + (bias ? __ldg(bias + e) : 0.0f);
            }
        }
        // lane e (< n) ranks its own expert: rank = number of experts ahead of it
        // (a larger logit, or an equal logit at a lower index).
        float mine = 0.0f, lmax = -INFINITY;
#pragma unroll
        for (int e = 0; e < NMAX; ++e) {
            if (e < n) {
                if (e == lane) mine = acc[e];
                lmax = fmaxf(lmax, acc[e]);
            }
        }
        int rank = 0;
#pragma unroll
        for (int e = 0; e < NMAX; ++e) {
            if (e < n) rank += (acc[e] > mine) || (acc[e] == mine && e < lane);
        }
        const bool kept = lane < n && rank < K;
        // Softmax over the kept logits only (the others are -inf), shifted by the max.
        float num = kept ? expf(mine - lmax) : 0.0f;
        float z = num;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        if (kept) {
            topk_idx[static_cast<size_t>(t) * K + rank] = lane;
            topk_w[static_cast<size_t>(t) * K + rank] = num / z;
        }
        if (logits_out && lane < n) logits_out[static_cast<size_t>(t) * n + lane] = mine;
    }
}

template <typename TX, int NMAX>
static cudaError_t launch_router_t(const void* x, const float* Wg, const float* bias, int T, int d,
                                   int n, int K, int32_t* idx, float* w, float* logits, int num_sms,
                                   cudaStream_t s) {
    const int threads = 512, warps = threads / 32;
    const size_t smem = static_cast<size_t>(n) * d * sizeof(float);
    auto kern = router_topk_kernel<TX, NMAX>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    int blocks = (T + warps - 1) / warps;
    if (blocks > num_sms) blocks = num_sms;
    if (blocks < 1) blocks = 1;
    kern<<<blocks, threads, smem, s>>>(static_cast<const TX*>(x), Wg, bias, T, d, n, K, idx, w, logits);
    return cudaGetLastError();
}

cudaError_t launch_router(ElemType et, const void* x, const float* Wg, const float* bias, int T, int d,
                          int n, int K, int32_t* idx, float* w, float* logits, int num_sms,
                          cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    if (et == ElemType::BF16) {
        if (n <= 8) return launch_router_t<__nv_bfloat16, 8>(x, Wg, bias, T, d, n, K, idx, w, logits, num_sms, s);
        if (n <= 16) return launch_router_t<__nv_bfloat16, 16>(x, Wg, bias, T, d, n, K, idx, w, logits, num_sms, s);
        return launch_router_t<__nv_bfloat16, 32>(x, Wg, bias, T, d, n, K, idx, w, logits, num_sms, s);
    }
    if (n <= 8) return launch_router_t<float, 8>(x, Wg, bias, T, d, n, K, idx, w, logits, num_sms, s);
    if (n <= 16) return launch_router_t<float, 16>(x, Wg, bias, T, d, n, K, idx, w, logits, num_sms, s);
    return launch_router_t<float, 32>(x, Wg, bias, T, d, n, K, idx, w, logits, num_sms, s);
}

// ---------------------------------------------------------------------------
// Dispatch, one block of 1024 threads.  Thread i owns the contiguous run
// [i*C, (i+1)*C) of flat assignments a = t*K + slot.  (1) per-thread expert
// histogram; (2) exclusive scan in (expert, thread) order, which is the
// stable order; (3) each thread scatters its run in order:
//   perm[pos] = a, inv[a] = pos.
// Same input -> same output, with no atomics on the data path.
constexpr int kDispatchThreads = 1024;

__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int ws = warp_sums[lane];
        int wi = ws;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += o;
        }
        warp_sums[lane] = wi - ws;   // exclusive prefix of warp totals
        if (lane == 31) warp_sums[32] = wi;
    }
    __syncthreads();
    int excl = incl - v + warp_sums[warp];
    total = warp_sums[32];
    __syncthreads();
    return excl;
}

__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(const int32_t* __restrict__ topk_idx,
                                                                    int R, int n, int* __restrict__ sched,
                                                                    int32_t* __restrict__ perm,
                                                                    int32_t* __restrict__ inv,
                                                                    KStatus st) {
    extern __shared__ int hist[];   // [n][kDispatchThreads]
    __shared__ int warp_sums[33];
    __shared__ int s_off[33];
    const int tid = threadIdx.x;
    const int C = (R + kDispatchThreads - 1) / kDispatchThreads;
    const int a0 = min(R, tid * C), a1 = min(R, a0 + C);
    for (int e = 0; e < n; ++e) hist[e * kDispatchThreads + tid] = 0;
    bool bad = false;
    for (int a = a0; a < a1; ++a) {
        int e = topk_idx[a];
        if (e < 0 || e >= n) { bad = true; continue; }
        hist[e * kDispatchThreads + tid] += 1;
    }
    if (bad) report(st, kStatusBounds);
    __syncthreads();
    int running = 0;
    for (int e = 0; e < n; ++e) {
        int total;
        int excl = block_exclusive_scan(hist[e * kDispatchThreads + tid], warp_sums, total);
        hist[e * kDispatchThreads + tid] = excl;
        if (tid == 0) {
            sched[e] = total;
            sched[n + e] = running;
            s_off[e] = running;
        }
        running += total;
    }
    if (tid == 0) {
        sched[2 * n] = running;
        int tp = 0;
        for (int e = 0; e < n; ++e) {
            sched[2 * n + 1 + e] = tp;
            tp += (sched[e] + kTileM - 1) / kTileM;
        }
        sched[3 * n + 1] = tp;
    }
    __syncthreads();
    for (int a = a0; a < a1; ++a) {
        int e = topk_idx[a];
        if (e < 0 || e >= n) continue;
        int pos = s_off[e] + hist[e * kDispatchThreads + tid]++;
        perm[pos] = a;
        inv[a] = pos;
    }
}

cudaError_t launch_dispatch(const int32_t* topk_idx, int R, int n, int* sched, int32_t* perm,
                            int32_t* inv, KStatus st, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(n) * kDispatchThreads * sizeof(int);
    cudaError_t err = cudaFuncSetAttribute(dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    dispatch_kernel<<<1, kDispatchThreads, smem, s>>>(topk_idx, R, n, sched, perm, inv, st);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Row gather: Xp[pos][:] = x[perm[pos] / K][:], one warp per row, 16-byte moves.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ perm, int R,
                                                          int K, int row_vecs, uint4* __restrict__ Xp) {
    const int lane = threadIdx.x & 31;
    for (int pos = blockIdx.x * 8 + (threadIdx.x >> 5); pos < R; pos += gridDim.x * 8) {
        const int t = perm[pos] / K;
        const uint4* src = x + static_cast<size_t>(t) * row_vecs;
        uint4* dst = Xp + static_cast<size_t>(pos) * row_vecs;
        for (int v = lane; v < row_vecs; v += 32) dst[v] = __ldg(src + v);
    }
}

cudaError_t launch_gather(ElemType et, const void* x, const int32_t* perm, int R, int K, int d, void* Xp,
                          cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    const int row_bytes = d * (et == ElemType::BF16 ? 2 : 4);
    const int row_vecs = row_bytes / 16;
    int blocks = (R + 7) / 8;
    if (blocks > 4096) blocks = 4096;
    gather_rows_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint4*>(x), perm, R, K, row_vecs,
                                              static_cast<uint4*>(Xp));
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Combine: y[t][i] = sum_{k=0}^{K-1} Ys[t*K+k][i], added in slot order in fp32
// and rounded once to the output type.  Ys rows already carry the gate weight.
template <typename TY>
__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ Ys, int T, int K, int d4,
                                                      TY* __restrict__ y) {
    const size_t total = static_cast<size_t>(T) * d4;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t t = i / d4, c = i % d4;
        const float4* src = Ys + t * K * d4 + c;
        float4 a = __ldg(src);
        for (int k = 1; k < K; ++k) {
            float4 b = __ldg(src + static_cast<size_t>(k) * d4);
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
        }
        if constexpr (sizeof(TY) == 4) {
            reinterpret_cast<float4*>(y)[i] = a;
        } else {
            uint2 o;
            o.x = pack_bf16x2(a.x, a.y);
            o.y = pack_bf16x2(a.z, a.w);
            reinterpret_cast<uint2*>(y)[i] = o;
        }
    }
}

cudaError_t launch_combine(ElemType et, const float* Ys, int T, int K, int d, void* y, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int d4 = d / 4;
    const size_t total = static_cast<size_t>(T) * d4;
    int blocks = static_cast<int>((total + 255) / 256);
    if (blocks > 148 * 16) blocks = 148 * 16;
    if (et == ElemType::BF16)
        combine_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(Ys), T, K,
                                                             d4, static_cast<__nv_bfloat16*>(y));
    else
        combine_kernel<float><<<blocks, 256, 0, s>>>(reinterpret_cast<const float4*>(Ys), T, K, d4,
                                                     static_cast<float*>(y));
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Bounded-wait self-test: thread 0 waits on an mbarrier that nothing ever
// arrives on; the wait gives up after st.wait_ns and records a timeout.
__global__ void wait_selftest_kernel(KStatus st) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_barrier_init();
        if (!mbar_wait(smem_u32(&bar), 0, st, nullptr)) report(st, kStatusTimeout);
    }
}

cudaError_t launch_wait_selftest(KStatus st, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(st);
    return cudaGetLastError();
}

}  // namespace moe
