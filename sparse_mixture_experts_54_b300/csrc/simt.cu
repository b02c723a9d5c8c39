// simt.cu -- grouped expert GEMMs on CUDA cores (fp32 FMA, no TF32), used for
// the fp32 element type, whose parity bar (1e-5 relative) rules out tensor-core
// fp32 modes.  Same math as the tensor-core path:
//   H[r][f]  = SiLU(sum_j Xp[r][j] W1[e][f][j]) * (sum_j Xp[r][j] W3[e][f][j])
//   Ys[a][i] = g_a * sum_f H[r][f] W2[e][i][f],   a = perm[r]
// (SwiGLU expert and gate-weighted output: aiqianji 3.2.4, code block D.)
// Rows r of expert e are offsets[e] .. offsets[e]+counts[e]-1 (expert-contiguous).
#include "kernels.h"

namespace moe {

constexpr int SB_M = 64, SB_N = 64, SB_K = 16;   // block tile; 16x16 threads, 4x4 outputs each

// Which expert and which M-block of it this block works on, for an SB_M tiling.
__device__ __forceinline__ bool simt_tile(const int* sched, int n, int mt, int& e, int& row0, int& rend) {
    int acc = 0;
    for (int k = 0; k < n; ++k) {
        const int c = sched[k];
        const int tiles = (c + SB_M - 1) / SB_M;
        if (mt < acc + tiles) {
            e = k;
            row0 = sched[n + k] + (mt - acc) * SB_M;
            rend = sched[n + k] + c;
            return true;
        }
        acc += tiles;
    }
    return false;
}

template <typename TX>
__global__ void __launch_bounds__(256) simt_gemm13_kernel(const TX* __restrict__ Xp, const TX* __restrict__ W1,
                                                          const TX* __restrict__ W3, TX* __restrict__ H,
                                                          const int* __restrict__ sched, int n, int d, int F) {
    griddep_launch_dependents();
    griddep_wait();
    int e, row0, rend;
    if (!simt_tile(sched, n, blockIdx.x, e, row0, rend)) return;
    const int f0 = blockIdx.y * SB_N;
    __shared__ float xs[SB_K][SB_M + 4];
    __shared__ float w1s[SB_K][SB_N + 4];
    __shared__ float w3s[SB_K][SB_N + 4];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float a[4][4] = {}, b[4][4] = {};
    const TX* W1e = W1 + static_cast<size_t>(e) * F * d;
    const TX* W3e = W3 + static_cast<size_t>(e) * F * d;
    for (int k0 = 0; k0 < d; k0 += SB_K) {
        for (int i = threadIdx.x; i < SB_M * SB_K; i += 256) {
            const int r = i / SB_K, kk = i % SB_K;
            const int row = row0 + r, k = k0 + kk;
            xs[kk][r] = (row < rend && k < d) ? to_f32(Xp[static_cast<size_t>(row) * d + k]) : 0.0f;
            const int f = f0 + r;
            const bool okw = f < F && k < d;
            w1s[kk][r] = okw ? to_f32(W1e[static_cast<size_t>(f) * d + k]) : 0.0f;
            w3s[kk][r] = okw ? to_f32(W3e[static_cast<size_t>(f) * d + k]) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SB_K; ++kk) {
            float xv[4], v1[4], v3[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                xv[u] = xs[kk][ty * 4 + u];
                v1[u] = w1s[kk][tx * 4 + u];
                v3[u] = w3s[kk][tx * 4 + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    a[u][v] = fmaf(xv[u], v1[v], a[u][v]);
                    b[u][v] = fmaf(xv[u], v3[v], b[u][v]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int row = row0 + ty * 4 + u;
        if (row >= rend) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int f = f0 + tx * 4 + v;
            if (f < F) H[static_cast<size_t>(row) * F + f] = from_f32<TX>(silu_f(a[u][v]) * b[u][v]);
        }
    }
}

template <typename TX>
__global__ void __launch_bounds__(256) simt_gemm2_kernel(const TX* __restrict__ H, const TX* __restrict__ W2,
                                                         float* __restrict__ Ys, const int* __restrict__ sched,
                                                         const int32_t* __restrict__ perm,
                                                         const float* __restrict__ topk_w, int n, int d, int F) {
    griddep_launch_dependents();
    griddep_wait();
    int e, row0, rend;
    if (!simt_tile(sched, n, blockIdx.x, e, row0, rend)) return;
    const int i0 = blockIdx.y * SB_N;
    __shared__ float hs[SB_K][SB_M + 4];
    __shared__ float ws[SB_K][SB_N + 4];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float o[4][4] = {};
    const TX* W2e = W2 + static_cast<size_t>(e) * d * F;
    for (int k0 = 0; k0 < F; k0 += SB_K) {
        for (int i = threadIdx.x; i < SB_M * SB_K; i += 256) {
            const int r = i / SB_K, kk = i % SB_K;
            const int row = row0 + r, k = k0 + kk;
            hs[kk][r] = (row < rend && k < F) ? to_f32(H[static_cast<size_t>(row) * F + k]) : 0.0f;
            const int oi = i0 + r;
            ws[kk][r] = (oi < d && k < F) ? to_f32(W2e[static_cast<size_t>(oi) * F + k]) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SB_K; ++kk) {
            float hv[4], wv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                hv[u] = hs[kk][ty * 4 + u];
                wv[u] = ws[kk][tx * 4 + u];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v) o[u][v] = fmaf(hv[u], wv[v], o[u][v]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int row = row0 + ty * 4 + u;
        if (row >= rend) continue;
        const int a = perm[row];
        const float g = topk_w[a];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const int oi = i0 + tx * 4 + v;
            if (oi < d) Ys[static_cast<size_t>(a) * d + oi] = g * o[u][v];
        }
    }
}

static int simt_max_mtiles(int R, int n) { return (R + SB_M - 1) / SB_M + n; }

cudaError_t launch_simt_gemm13(ElemType et, const void* Xp, const void* W1, const void* W3, void* H,
                               const int* sched, int n, int d, int F, int R, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    dim3 grid(simt_max_mtiles(R, n), (F + SB_N - 1) / SB_N);
    if (et == ElemType::F32)
        return launch_pdl(simt_gemm13_kernel<float>, grid, dim3(256), 0, s, static_cast<const float*>(Xp),
                          static_cast<const float*>(W1), static_cast<const float*>(W3), static_cast<float*>(H), sched,
                          n, d, F);
    return launch_pdl(simt_gemm13_kernel<__nv_bfloat16>, grid, dim3(256), 0, s,
                      static_cast<const __nv_bfloat16*>(Xp), static_cast<const __nv_bfloat16*>(W1),
                      static_cast<const __nv_bfloat16*>(W3), static_cast<__nv_bfloat16*>(H), sched, n, d, F);
}

cudaError_t launch_simt_gemm2(ElemType et, const void* H, const void* W2, float* Ys, const int* sched,
                              const int32_t* perm, const float* topk_w, int n, int d, int F, int R,
                              cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    dim3 grid(simt_max_mtiles(R, n), (d + SB_N - 1) / SB_N);
    if (et == ElemType::F32)
        return launch_pdl(simt_gemm2_kernel<float>, grid, dim3(256), 0, s, static_cast<const float*>(H),
                          static_cast<const float*>(W2), Ys, sched, perm, topk_w, n, d, F);
    return launch_pdl(simt_gemm2_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, static_cast<const __nv_bfloat16*>(H),
                      static_cast<const __nv_bfloat16*>(W2), Ys, sched, perm, topk_w, n, d, F);
}

}  // namespace moe
