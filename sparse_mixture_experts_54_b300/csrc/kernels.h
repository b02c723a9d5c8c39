// kernels.h -- host-side launchers of the MoE kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "combine_epi.cuh"
#include "common.cuh"

namespace moe {

// Schedule block written by the dispatch kernel (int32, device):
//   [0, n)          counts[e]
//   [n, 2n+1)       offsets[e] (exclusive scan), offsets[n] = R
//   [2n+1, 3n+2)    tile_prefix[e] = sum_{e'<e} ceil(counts[e'] / kTileM), tile_prefix[n] = total
constexpr int kTileM = 128;
inline int sched_ints(int n) { return 3 * n + 2; }

enum class ElemType { BF16 = 0, F32 = 1 };

// Row blocks per tile group of the grouped GEMMs: as many as keep the group's A
// rows (rows x k_elems bf16 each) within 96 MB, most of the 126 MB L2.
inline int tile_group_rows(int rows_per_block, int k_elems) {
    const long long bytes = static_cast<long long>(rows_per_block) * k_elems * 2;
    const long long g = (96ll << 20) / (bytes > 0 ? bytes : 1);
    return g < 1 ? 1 : static_cast<int>(g);
}

// Launch with programmatic stream serialisation (see griddep_wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// routing ---------------------------------------------------------------------
cudaError_t launch_router(ElemType et, const void* x, const float* Wg, const float* bias, int T, int d,
                          int n, int K, int32_t* topk_idx, float* topk_w, float* logits, int num_sms,
                          cudaStream_t s);
cudaError_t launch_dispatch(const int32_t* topk_idx, int R, int n, int* sched, int32_t* perm,
                            int32_t* inv, KStatus st, cudaStream_t s);
cudaError_t launch_gather(ElemType et, const void* x, const int32_t* perm, int R, int K, int d,
                          void* Xp, cudaStream_t s);
// resid: optional [T][d] (may be y) added to the slot sum before the rounding.
cudaError_t launch_combine(ElemType et, const float* Ys, int T, int K, int d, const void* resid, void* y,
                           cudaStream_t s);

// Router + top-k + dispatch + row gather in one kernel (route_fused.cu).  xchg
// holds fused_route_xchg_ints() ints that must be zero before the first call;
// every complete call leaves its barrier words as it found them (the ready word
// is cleared at the start of every call).  Xp and logits may be null.
// rstd non-null ([T] floats): RMSNorm the rows first (eps = norm_eps).
constexpr int kFusedRouteMaxBlocks = 160;
// The word after the block counts is the schedule-ready word of the decode
// kernels (cleared by the routing kernel of every call).
constexpr int kReadyWord = 2 + kFusedRouteMaxBlocks * 32;
inline int fused_route_xchg_ints() { return kReadyWord + 1; }
int fused_route_blocks(int T, int num_sms);
cudaError_t launch_fused_route(ElemType et, const void* x, const float* Wg, const float* bias, int T, int d, int n,
                               int K, int32_t* topk_idx, float* topk_w, float* logits, int* sched, int32_t* perm,
                               int32_t* inv, void* Xp, int* xchg, float norm_eps, float* rstd, KStatus st,
                               int num_sms, cudaStream_t s);

// CUDA-core grouped GEMMs (fp32 path) ------------------------------------------
cudaError_t launch_simt_gemm13(ElemType et, const void* Xp, const void* W1, const void* W3, void* H,
                               const int* sched, int n, int d, int F, int R, cudaStream_t s);
cudaError_t launch_simt_gemm2(ElemType et, const void* H, const void* W2, float* Ys, const int* sched,
                              const int32_t* perm, const float* topk_w, int n, int d, int F, int R,
                              cudaStream_t s);

// tcgen05 grouped GEMMs (bf16 path) --------------------------------------------
bool encode_map_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows);
cudaError_t launch_tc_gemm13(const CUtensorMap& mapXp, const CUtensorMap& mapW1,
                             const CUtensorMap& mapW3, const int* sched, int n, int d, int F, int R,
                             __nv_bfloat16* H, KStatus st, int num_sms, cudaStream_t s);
// comb.cnt non-null: the epilogue also does the combine (combine_epi.cuh) and writes y.
cudaError_t launch_tc_gemm2(const CUtensorMap& mapH, const CUtensorMap& mapW2, const int* sched, int n,
                            int d, int F, int R, float* Ys, const int32_t* perm, const float* topk_w,
                            const CombineArgs& comb, KStatus st, int num_sms, cudaStream_t s);

// tcgen05 grouped GEMMs on CTA pairs (cta_group::2; 256-row tiles) -------------
bool pair_gemm_available(int num_sms);
// mapW1/mapW3: 128-row boxes; mapW1_64/mapW3_64: the same tensors with 64-row boxes.
cudaError_t launch_pair_gemm13(const CUtensorMap& mapXp, const CUtensorMap& mapW1, const CUtensorMap& mapW3,
                               const CUtensorMap& mapW1_64, const CUtensorMap& mapW3_64, const int* sched, int n,
                               int d, int F, int R, __nv_bfloat16* H, KStatus st, int num_sms, cudaStream_t s);
cudaError_t launch_pair_gemm2(const CUtensorMap& mapH, const CUtensorMap& mapW2_128, const int* sched, int n, int d,
                              int F, int R, float* Ys, const int32_t* perm, const float* topk_w,
                              const CombineArgs& comb, KStatus st, int num_sms, cudaStream_t s);

// weight-streaming decode path (bf16, small T) ----------------------------------
constexpr int kDecodeMaxT = 256;     // tokens per call the decode kernels accept
constexpr int kDecodeMaxSplits = 16;

// Sum of the S (<= kDecodeMaxSplits) K-split partials p[s * stride], added in
// s order.  The loads are issued eight at a time before their adds, so a small
// batch's few threads wait for S/8 round trips to L2 instead of S in a row.
__device__ __forceinline__ float4 sum_splits(const float4* __restrict__ p, size_t stride, int S) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (s0 + j < S) v[j] = __ldg(p + static_cast<size_t>(s0 + j) * stride);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (s0 + j == 0) {
                a = v[0];
            } else if (s0 + j < S) {
                a.x += v[j].x;
                a.y += v[j].y;
                a.z += v[j].z;
                a.w += v[j].w;
            }
        }
    }
    return a;
}

// Two such sums at once, of S0 and S1 splits, their loads issued together (each
// still in s order), kBatch splits of each per round trip.
template <int kBatch = 8>
__device__ __forceinline__ void sum_splits_pair(const float4* __restrict__ p, const float4* __restrict__ q,
                                                size_t stride, int S0, int S1, float4& a, float4& b) {
    a = b = make_float4(0.f, 0.f, 0.f, 0.f);
    const int S = S0 > S1 ? S0 : S1;
    for (int s0 = 0; s0 < S; s0 += kBatch) {
        float4 u[kBatch], v[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (s0 + j < S0) u[j] = __ldg(p + static_cast<size_t>(s0 + j) * stride);
            if (s0 + j < S1) v[j] = __ldg(q + static_cast<size_t>(s0 + j) * stride);
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
            if (s0 + j == 0) {
                a = u[0];
                b = v[0];
            } else {
                if (s0 + j < S0) {
                    a.x += u[j].x; a.y += u[j].y; a.z += u[j].z; a.w += u[j].w;
                }
                if (s0 + j < S1) {
                    b.x += v[j].x; b.y += v[j].y; b.z += v[j].z; b.w += v[j].w;
                }
            }
        }
    }
}

// How the weight-streaming kernels split K, and so which partial-sum slots the
// SwiGLU and combine kernels add for a row block.
//
// Uniform (sk == 0): item it = (unit, split) with the split fastest; a unit is
// (touched expert, row block of 128 output features) in expert order; split sp
// covers k-blocks [sp kb / S, (sp + 1) kb / S) and writes slot sp.
//
// Stream-K (sk != 0): the k-blocks of all U units laid end to end, W = U kb, and
// CTA c of the first G takes [c W / G, (c + 1) W / G) in order, so every CTA
// streams the same number of weight bytes (to one k-block) and none waits for a
// last, partly filled wave.  A unit's k-blocks fall to consecutive CTAs; the CTA
// holding a piece writes slot (its index - the index of the CTA that holds the
// unit's first k-block), slots 0 .. n_u - 1 in K order.  G is the grid cut so
// that every CTA's share is at least kb / (kDecodeMaxSplits - 1) k-blocks, hence
// n_u <= kDecodeMaxSplits.
struct SplitGeom {
    int sk = 0;               // 0 uniform, 1 stream-K
    int S = 1;                // uniform: splits
    int kb = 1;               // k-blocks per unit
    int rb = 1;               // row blocks (of 128 output features) per expert
    int grid = 1;             // CTAs of the weight-streaming launch
    const int* sched = nullptr;   // stream-K: the call's schedule (counts first)
    int n = 1;                // experts
};
__device__ __forceinline__ long long sk_start(int c, long long W, int G) {
    return static_cast<long long>(c) * W / G;
}
// the CTA whose share holds flat k-block x (32-bit division whenever it fits)
__device__ __forceinline__ int sk_cta_of(long long x, long long W, int G) {
    const unsigned long long num = static_cast<unsigned long long>(x + 1) * G + static_cast<unsigned long long>(W) - 1;
    if (num < (1ull << 32)) return static_cast<int>(static_cast<unsigned>(num) / static_cast<unsigned>(W)) - 1;
    return static_cast<int>(num / static_cast<unsigned long long>(W)) - 1;
}
__device__ __forceinline__ int sk_grid(long long W, int kb, int grid) {
    const long long m = (kb + kDecodeMaxSplits - 2) / (kDecodeMaxSplits - 1);
    long long g = W / m;
    if (g > grid) g = grid;
    return g < 1 ? 1 : static_cast<int>(g);
}
// slots holding unit u's partial sums
__device__ __forceinline__ int sk_slots(int u, long long W, int kb, int G) {
    return sk_cta_of(static_cast<long long>(u + 1) * kb - 1, W, G) - sk_cta_of(static_cast<long long>(u) * kb, W, G) +
           1;
}

int decode_pick_splits(int units, int kblocks, int num_sms);
// ready (may be null): the schedule-ready word (xchg + kReadyWord) of the
// routing kernel that ran first in the call; the W1/W3 kernel sets it and the W2
// kernel then sends its first weight tiles before waiting on the SwiGLU kernel.
// splits: uniform K splits, or 0 for stream-K.  The SwiGLU and combine
// launches take the geometry of the launch that wrote their partial sums
// (decode_geom), and the combine the assignments' experts (topk_idx) to find a
// row's unit under stream-K.
cudaError_t launch_decode_w13(const CUtensorMap& mapW1, const CUtensorMap& mapW3, const CUtensorMap& mapXp32,
                              const int* sched, int n, int d, int F, int T, int K, int splits, float* Pa, float* Pb,
                              KStatus st, int num_sms, cudaStream_t s, int* ready = nullptr);
cudaError_t launch_decode_w2(const CUtensorMap& mapW2_128, const CUtensorMap& mapH32, const int* sched, int n, int d,
                             int F, int T, int K, int splits, float* P2, KStatus st, int num_sms, cudaStream_t s,
                             int* ready = nullptr);
SplitGeom decode_geom(int splits, int kblocks, int row_blocks, const int* sched, int n, int num_sms);
cudaError_t launch_decode_swiglu(const float* Pa, const float* Pb, const SplitGeom& g, int R, int F, __nv_bfloat16* H,
                                 cudaStream_t s);
cudaError_t launch_decode_combine(ElemType et, const float* P2, const SplitGeom& g, int R, const int32_t* inv,
                                  const int32_t* topk_idx, const float* topk_w, int T, int K, int d, const void* resid,
                                  void* y, cudaStream_t s);

// the same with e4m3 weights and fp32 row scales (decode_fp8.cu); the weight
// maps come from encode_map_u8_sw64, the partial sums feed launch_decode_swiglu /
// launch_decode_combine unchanged
bool encode_map_u8_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols);
cudaError_t launch_decode_fp8_w13(const CUtensorMap& mapW1q, const CUtensorMap& mapW3q, const CUtensorMap& mapXp32,
                                  const float* W1s, const float* W3s, const int* sched, int n, int d, int F, int T,
                                  int K, int splits, float* Pa, float* Pb, KStatus st, int num_sms, cudaStream_t s);
cudaError_t launch_decode_fp8_w2(const CUtensorMap& mapW2q, const CUtensorMap& mapH32, const float* W2s,
                                 const int* sched, int n, int d, int F, int T, int K, int splits, float* P2, KStatus st,
                                 int num_sms, cudaStream_t s);

// the same with e4m3 weights multiplied by the e4m3 tensor-core MMA
// (decode_fp8_mma.cu): token rows split into hi/lo e4m3 rows with a
// power-of-two scale per row; weight maps from encode_map_u8_sw128 (128-row
// boxes), token maps with 64-row boxes; partial sums as above
bool encode_map_u8_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
cudaError_t launch_split_rows_e4m3(const __nv_bfloat16* X, int R, int d, uint8_t* Xq, float* xinv, cudaStream_t s);
// chunks: the W2 GEMM's K splits (one H scale per row and split); hinv [chunks][R]
cudaError_t launch_decode_swiglu_split(const float* Pa, const float* Pb, int S, int R, int F, int chunks, uint8_t* Hq,
                                       float* hinv, cudaStream_t s);
cudaError_t launch_decode_f8_w13(const CUtensorMap& mapW1q, const CUtensorMap& mapW3q, const CUtensorMap& mapXq,
                                 const float* W1s, const float* W3s, const float* xinv, const int* sched, int n, int d,
                                 int F, int T, int K, int splits, float* Pa, float* Pb, KStatus st, int num_sms,
                                 cudaStream_t s);
cudaError_t launch_decode_f8_w2(const CUtensorMap& mapW2q, const CUtensorMap& mapHq, const float* W2s,
                                const float* hinv, const int* sched, int n, int d, int F, int T, int K, int splits,
                                float* P2, KStatus st, int num_sms, cudaStream_t s);

// self-test of the bounded waits -------------------------------------------------
cudaError_t launch_wait_selftest(KStatus st, cudaStream_t s);

}  // namespace moe
