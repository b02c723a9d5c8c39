// route.cu -- router logits + top-k gate, deterministic dispatch, row gather,
// and the fixed-order combine of each token's expert rows.
//
// Router: G(x) = Softmax(TopK(x . W_g)), TopK keeping the K largest logits
// (Mixtral of Experts section 2.1, restated in aiqianji section 2.1.1; router
// is nn.Linear(hidden_dim, num_experts, bias=False), aiqianji 2.1.4).
// Dispatch replaces the one_hot/permute/where walk and the row gather of
// aiqianji 3.1.2 (code blocks B, C); combine replaces index_add_ there.
#include "kernels.h"
#include "route_common.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// Router for small batches: one block of 8 warps per token.  Warp w sums the
// 8-element chunks w, w+8, w+16, ... of the row (lane-strided), reduces them
// with a butterfly, and warp 0 adds the 8 warp sums in warp order, so the
// result is fixed for a given d.  All loads of a lane are issued before use.
template <typename TX, int NMAX>
__global__ void __launch_bounds__(256) router_small_kernel(const TX* __restrict__ x, const float* __restrict__ Wg,
                                                          const float* __restrict__ bias, int d, int n, int K,
                                                          int32_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_w,
                                                          float* __restrict__ logits_out) {
    __shared__ float part[8][NMAX];
    griddep_launch_dependents();
    griddep_wait();
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const TX* xr = x + static_cast<size_t>(t) * d;
    float acc[NMAX];
#pragma unroll
    for (int e = 0; e < NMAX; ++e) acc[e] = 0.0f;
    const int nchunks = d / 8;
    for (int c0 = warp + 8 * lane; c0 < nchunks; c0 += 8 * 32 * 2) {
        float xv[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) load8(xr, (c0 + u * 256) * 8, d, xv[u]);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int j0 = (c0 + u * 256) * 8;
            if (j0 >= d) break;
#pragma unroll
            for (int e = 0; e < NMAX; ++e)
                if (e < n) {
                    const float* w = Wg + static_cast<size_t>(e) * d + j0;
                    float wv[8];
                    float4 w0 = __ldg(reinterpret_cast<const float4*>(w));
                    float4 w1 = __ldg(reinterpret_cast<const float4*>(w + 4));
                    wv[0] = w0.x; wv[1] = w0.y; wv[2] = w0.z; wv[3] = w0.w;
                    wv[4] = w1.x; wv[5] = w1.y; wv[6] = w1.z; wv[7] = w1.w;
                    float a = acc[e];
#pragma unroll
                    for (int q = 0; q < 8; ++q) a = fmaf(xv[u][q], wv[q], a);
                    acc[e] = a;
                }
        }
    }
#pragma unroll
    for (int e = 0; e < NMAX; ++e) {
        if (e < n) {
            float v = acc[e];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) part[warp][e] = v;
        }
    }
    __syncthreads();
    if (warp != 0) return;
    float l[NMAX];
#pragma unroll
    for (int e = 0; e < NMAX; ++e) {
        float v = 0.0f;
        if (e < n) {
#pragma unroll
            for (int w = 0; w < 8; ++w) v += part[w][e];
            v += bias ? __ldg(bias + e) : 0.0f;
        }
        l[e] = v;
    }
    topk_gate_write<NMAX>(l, n, K, t, lane, topk_idx, topk_w, logits_out);
}

// ---------------------------------------------------------------------------
// Router for large batches: W_g [n][d] fp32 is staged once per block in shared
// memory, and each warp routes kTokPerWarp tokens at a time so that every
// W_g value read from shared memory serves all of them.  Lane l owns the
// 8-element chunks l, l+32, l+64, ... of a row and accumulates them in that
// order; the warp adds the lanes with a butterfly, so every lane holds all n
// logits of each token and the result does not depend on timing.
constexpr int kTokPerWarp = 4;

template <typename TX, int NMAX>
__global__ void __launch_bounds__(256) router_topk_kernel(const TX* __restrict__ x,
                                                          const float* __restrict__ Wg,
                                                          const float* __restrict__ bias, int T,
                                                          int d, int n, int K,
                                                          int32_t* __restrict__ topk_idx,
                                                          float* __restrict__ topk_w,
                                                          float* __restrict__ logits_out) {
    extern __shared__ float wg_s[];
    griddep_launch_dependents();
    {
        // Stage W_g with 8 independent 16-byte loads in flight per thread.  This
        // prologue may overlap the previous kernel: no kernel of the layer writes W_g.
        const int total4 = n * d / 4, stride = blockDim.x;
        const float4* src = reinterpret_cast<const float4*>(Wg);
        float4* dst = reinterpret_cast<float4*>(wg_s);
        for (int i0 = threadIdx.x; i0 < total4; i0 += 8 * stride) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * stride;
                v[u] = i < total4 ? __ldg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * stride;
                if (i < total4) dst[i] = v[u];
            }
        }
    }
    griddep_wait();
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int groups = (T + kTokPerWarp - 1) / kTokPerWarp;
    for (int g = blockIdx.x * warps + (threadIdx.x >> 5); g < groups; g += gridDim.x * warps) {
        const int t0 = g * kTokPerWarp;
        float acc[kTokPerWarp][NMAX];
#pragma unroll
        for (int q = 0; q < kTokPerWarp; ++q)
#pragma unroll
            for (int e = 0; e < NMAX; ++e) acc[q][e] = 0.0f;
        for (int j0 = lane * 8; j0 < d; j0 += 256) {
            float xv[kTokPerWarp][8];
#pragma unroll
            for (int q = 0; q < kTokPerWarp; ++q) {
                const int t = min(t0 + q, T - 1);   // tail tokens repeat the last row; not written
                load8(x + static_cast<size_t>(t) * d, j0, d, xv[q]);
            }
#pragma unroll
            for (int e = 0; e < NMAX; ++e) {
                if (e < n) {
                    const float* w = wg_s + e * d + j0;
                    const float4 w0 = *reinterpret_cast<const float4*>(w);
                    const float4 w1 = *reinterpret_cast<const float4*>(w + 4);
                    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int q = 0; q < kTokPerWarp; ++q) {
                        float a = acc[q][e];
#pragma unroll
                        for (int u = 0; u < 8; ++u) a = fmaf(xv[q][u], wv[u], a);
                        acc[q][e] = a;
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kTokPerWarp; ++q) {
            // butterfly sum: identical result in every lane
#pragma unroll
            for (int e = 0; e < NMAX; ++e) {
                if (e < n) {
                    float v = acc[q][e];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    acc[q][e] = v + (bias ? __ldg(bias + e) : 0.0f);
                }
            }
            if (t0 + q < T) topk_gate_write<NMAX>(acc[q], n, K, t0 + q, lane, topk_idx, topk_w, logits_out);
        }
    }
}

// Batches up to this many tokens use the block-per-token router.
constexpr int kSmallRouterMaxT = 512;

template <typename TX, int NMAX>
static cudaError_t launch_router_t(const void* x, const float* Wg, const float* bias, int T, int d,
                                   int n, int K, int32_t* idx, float* w, float* logits, int num_sms,
                                   cudaStream_t s) {
    if (T <= kSmallRouterMaxT) {
        return launch_pdl(router_small_kernel<TX, NMAX>, dim3(T), dim3(256), 0, s, static_cast<const TX*>(x), Wg,
                          bias, d, n, K, idx, w, logits);
    }
    const int threads = 256, warps = threads / 32;
    const size_t smem = static_cast<size_t>(n) * d * sizeof(float);
    auto kern = router_topk_kernel<TX, NMAX>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const int groups = (T + kTokPerWarp - 1) / kTokPerWarp;
    int blocks = (groups + warps - 1) / warps;
    if (blocks > 2 * num_sms) blocks = 2 * num_sms;
    if (blocks < 1) blocks = 1;
    return launch_pdl(kern, dim3(blocks), dim3(threads), smem, s, static_cast<const TX*>(x), Wg, bias, T, d, n, K,
                      idx, w, logits);
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
// Dispatch, one block of 1024 threads (32 warps).
//  (1) counts[e]: shared-memory histogram of the flat assignments
//      a = t*K + slot (the totals do not depend on the order of the adds);
//  (2) offsets = exclusive scan of counts, and the 128-row tile prefix;
//  (3) stable scatter, 1024 assignments per round in flat order: lanes of a
//      warp holding the same expert find each other (match_any), a lane's rank
//      among them is the number of such lanes below it, and the per-(warp,
//      expert) counts are scanned across the 32 warps in warp order.  So
//      pos = offsets[e] + (earlier rounds) + (earlier warps) + (earlier lanes):
//      perm[pos] = a, inv[a] = pos, ascending a within every expert.
// Same input -> same output; no atomics touch the output order.
constexpr int kDispatchThreads = 1024;

__global__ void __launch_bounds__(kDispatchThreads) dispatch_kernel(const int32_t* __restrict__ topk_idx,
                                                                    int R, int n, int* __restrict__ sched,
                                                                    int32_t* __restrict__ perm,
                                                                    int32_t* __restrict__ inv,
                                                                    KStatus st) {
    __shared__ int s_count[32];
    __shared__ int s_off[33];
    __shared__ int s_run[32];            // assignments of expert e placed in earlier rounds
    __shared__ int wtab[32][33];         // [warp][expert]: count, then base, of this round
    griddep_launch_dependents();
    griddep_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < 32) {
        s_count[tid] = 0;
        s_run[tid] = 0;
    }
    __syncthreads();
    bool bad = false;
    for (int a = tid; a < R; a += kDispatchThreads) {
        const int e = topk_idx[a];
        if (e < 0 || e >= n) {
            bad = true;
            continue;
        }
        atomicAdd(&s_count[e], 1);
    }
    if (bad) report(st, kStatusBounds);
    __syncthreads();
    if (tid == 0) {
        int running = 0, tp = 0;
        for (int e = 0; e < n; ++e) {
            const int c = s_count[e];
            sched[e] = c;
            sched[n + e] = running;
            sched[2 * n + 1 + e] = tp;
            s_off[e] = running;
            running += c;
            tp += (c + kTileM - 1) / kTileM;
        }
        sched[2 * n] = running;
        sched[3 * n + 1] = tp;
    }
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int c0 = 0; c0 < R; c0 += kDispatchThreads) {
        const int a = c0 + tid;
        int e = a < R ? topk_idx[a] : -1;
        if (e >= n) e = -1;
        wtab[warp][lane] = 0;
        __syncwarp();
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & lt_mask);
        if (e >= 0 && rank == 0) wtab[warp][e] = __popc(same);
        __syncthreads();
        if (warp < n) {
            // warp index = expert; lane index = the warp whose count is scanned
            const int v = wtab[lane][warp];
            const int run = s_run[warp];
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            wtab[lane][warp] = run + incl - v;
            __syncwarp();
            if (lane == 31) s_run[warp] = run + incl;
        }
        __syncthreads();
        if (e >= 0) {
            const int pos = s_off[e] + wtab[warp][e] + rank;
            perm[pos] = a;
            inv[a] = pos;
        }
        __syncthreads();
    }
}

cudaError_t launch_dispatch(const int32_t* topk_idx, int R, int n, int* sched, int32_t* perm,
                            int32_t* inv, KStatus st, cudaStream_t s) {
    if (n > 32) return cudaErrorInvalidValue;
    return launch_pdl(dispatch_kernel, dim3(1), dim3(kDispatchThreads), 0, s, topk_idx, R, n, sched, perm, inv, st);
}

// ---------------------------------------------------------------------------
// Row gather: Xp[pos][:] = x[perm[pos] / K][:], one warp per row, 16-byte moves.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ perm, int R,
                                                          int K, int row_vecs, uint4* __restrict__ Xp) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    for (int pos = blockIdx.x * 8 + (threadIdx.x >> 5); pos < R; pos += gridDim.x * 8) {
        const int t = perm[pos] / K;
        const uint4* src = x + static_cast<size_t>(t) * row_vecs;
        uint4* dst = Xp + static_cast<size_t>(pos) * row_vecs;
        for (int v0 = lane; v0 < row_vecs; v0 += 32 * 8) {
            uint4 r[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int v = v0 + 32 * u;
                if (v < row_vecs) r[u] = __ldg(src + v);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int v = v0 + 32 * u;
                if (v < row_vecs) dst[v] = r[u];
            }
        }
    }
}

cudaError_t launch_gather(ElemType et, const void* x, const int32_t* perm, int R, int K, int d, void* Xp,
                          cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    const int row_bytes = d * (et == ElemType::BF16 ? 2 : 4);
    const int row_vecs = row_bytes / 16;
    int blocks = (R + 7) / 8;
    if (blocks > 4096) blocks = 4096;
    return launch_pdl(gather_rows_kernel, dim3(blocks), dim3(256), 0, s, static_cast<const uint4*>(x), perm, R, K,
                      row_vecs, static_cast<uint4*>(Xp));
}

// ---------------------------------------------------------------------------
// Combine: y[t][i] = sum_{k=0}^{K-1} Ys[t*K+k][i], added in slot order in fp32
// and rounded once to the output type.  Ys rows already carry the gate weight.
// With resid (may be y itself): y = resid + the slot sum, one rounding.
template <typename TY>
__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ Ys, int T, int K, int d4,
                                                      const TY* resid, TY* y) {
    griddep_launch_dependents();
    griddep_wait();
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
        if (resid) {
            float r[4];
            if constexpr (sizeof(TY) == 4) {
                const float4 h = reinterpret_cast<const float4*>(resid)[i];
                r[0] = h.x; r[1] = h.y; r[2] = h.z; r[3] = h.w;
            } else {
                const uint2 h = reinterpret_cast<const uint2*>(resid)[i];
                r[0] = __low2float(*reinterpret_cast<const __nv_bfloat162*>(&h.x));
                r[1] = __high2float(*reinterpret_cast<const __nv_bfloat162*>(&h.x));
                r[2] = __low2float(*reinterpret_cast<const __nv_bfloat162*>(&h.y));
                r[3] = __high2float(*reinterpret_cast<const __nv_bfloat162*>(&h.y));
            }
            a.x = r[0] + a.x; a.y = r[1] + a.y; a.z = r[2] + a.z; a.w = r[3] + a.w;
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

cudaError_t launch_combine(ElemType et, const float* Ys, int T, int K, int d, const void* resid, void* y,
                           cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const int d4 = d / 4;
    const size_t total = static_cast<size_t>(T) * d4;
    int blocks = static_cast<int>((total + 255) / 256);
    if (blocks > 148 * 16) blocks = 148 * 16;
    if (et == ElemType::BF16)
        return launch_pdl(combine_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, s,
                          reinterpret_cast<const float4*>(Ys), T, K, d4, static_cast<const __nv_bfloat16*>(resid),
                          static_cast<__nv_bfloat16*>(y));
    return launch_pdl(combine_kernel<float>, dim3(blocks), dim3(256), 0, s, reinterpret_cast<const float4*>(Ys), T, K,
                      d4, static_cast<const float*>(resid), static_cast<float*>(y));
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
