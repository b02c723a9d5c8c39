// gemm_tc.cu -- grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// The per-expert loop of the code walkthrough (aiqianji 3.1.2: for each expert,
// gather its tokens, run w1/w3/w2, index_add_ back) becomes two persistent
// kernels over the expert-contiguous rows built by dispatch:
//
//   MODE 0 (W1/W3 + SwiGLU):  H[r][f] = SiLU(Xp[r] . W1[e][f]) * (Xp[r] . W3[e][f])
//   MODE 1 (W2 + gate):       Ys[a][i] = g_a * (H[r] . W2[e][i]),   a = perm[r]
//
// (SwiGLU expert and in-expert gate scaling: aiqianji 3.2.4, code block D.)
//
// Tile: 128 rows of one expert x 256 accumulator columns, K in steps of 64
// (one 128-byte swizzle row of bf16).  MODE 0's 256 columns are 128 W1
// outputs followed by the 128 W3 outputs of the same features, so one
// accumulator holds both halves of the SwiGLU product.  MODE 1's 256 columns
// are 256 output features.  Tiles run expert by expert; inside an expert the
// 128-row blocks vary fastest, so CTAs running at the same time share weight
// slabs through L2 and each weight byte comes from HBM about once.
//
// Warp roles (6 warps): warp 0 lane 0 issues TMA loads into a 4-stage ring;
// warp 1 owns tensor memory (512 columns = two 256-column accumulators) and
// its lane 0 issues the MMAs; warps 2-5 read the accumulator (each warp its
// 32-lane quadrant), apply the epilogue and store.  Every wait is bounded;
// a wait that runs out raises an abort flag, records a timeout in the status
// word, and all roles unwind, drain in-flight copies and MMAs, free tensor
// memory and return.
#include <cudaTypedefs.h>

#include "combine_epi.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int BM = kTileM;                 // 128 rows per tile
constexpr int BK = 64;                     // K per stage (128 B of bf16)
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int B_ROWS = 256;
constexpr int B_BYTES = B_ROWS * BK * 2;   // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr int MAX_EXPERTS = 32;
constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1;   // full, empty, acc_full, acc_empty, drain
constexpr size_t SMEM_BYTES = 1024 /*alignment slack*/ + STAGES * STAGE_BYTES + NUM_BARS * 8 + 16 +
                              (3 * MAX_EXPERTS + 2) * 4;
}  // namespace

struct TcArgs {
    const int* sched;
    int n;
    int kblocks;          // K / BK
    int ntiles;           // N-tiles per expert
    int group_m;          // row blocks per tile group (see tc_decode_tile)
    int b_rows_per_e;     // rows of the B tensor per expert (F for MODE 0, d for MODE 1)
    __nv_bfloat16* H;     // MODE 0 output, [R][F]
    int ldH;
    float* Ys;            // MODE 1 output, [R][d] by flat assignment
    int ldY;
    const int32_t* perm;
    const float* topk_w;
    int w_policy;         // L2 policy of weight loads: 0 evict_first, 1 evict_normal, 2 evict_last
    CombineArgs comb;     // MODE 1: fused combine into y (comb.cnt null: Ys only)
    KStatus st;
};

// tile -> (expert, 128-row block, N block).  Tiles are expert-major; inside an
// expert its row blocks are taken group_m at a time, and within a group the N
// blocks go in order with the group's row blocks fastest.  A group's rows (the
// A band) are sized on the host to stay in L2 while every N block of the
// weights streams past them once; an expert with at most group_m row blocks
// (every expert of a uniform batch of a few thousand tokens) is one group.
__device__ __forceinline__ void tc_decode_tile(const int* prefix, int n, int ntiles, int group_m, int tile, int& e,
                                               int& mb, int& nb) {
    int k = 0;
    while (k + 1 < n && prefix[k + 1] * ntiles <= tile) ++k;
    const int mt = prefix[k + 1] - prefix[k];
    const int local = tile - prefix[k] * ntiles;
    const int g = local / (group_m * ntiles);
    const int mg = min(group_m, mt - g * group_m);
    const int r = local - g * group_m * ntiles;
    e = k;
    nb = r / mg;
    mb = g * group_m + r % mg;
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1, TcArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t tiles_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t* tiles_ptr = smem_raw + (tiles_u32 - raw_u32);
    uint64_t* bars = reinterpret_cast<uint64_t*>(tiles_ptr + STAGES * STAGE_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_sched = reinterpret_cast<int*>(tmem_slot + 4);

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = p.n;
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), EPI_THREADS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB0);
        if (MODE == 0) tma_prefetch_desc(&tmB1);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    // Everything above is prologue that touches no buffer of the layer; the
    // schedule and the activations come from the kernels before this one.
    griddep_wait();
    for (int i = threadIdx.x; i < 3 * n + 2; i += THREADS) s_sched[i] = p.sched[i];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int* counts = s_sched;
    const int* offsets = s_sched + n;
    const int* prefix = s_sched + 2 * n + 1;
    const int total = prefix[n] * p.ntiles;
    const KStatus st = p.st;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            const uint64_t pol_act = policy_evict_last();
            const uint64_t pol_w = p.w_policy == 0 ? policy_evict_first()
                                   : p.w_policy == 2 ? policy_evict_last() : policy_evict_normal();
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                int e, mb, nb;
                tc_decode_tile(prefix, n, p.ntiles, p.group_m, tile, e, mb, nb);
                const int arow = offsets[e] + mb * BM;
                const int brow = e * p.b_rows_per_e + nb * (MODE == 0 ? 128 : 256);
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, st, abort_flag)) { ok = false; break; }
                    const uint32_t a_dst = tiles_u32 + stage * STAGE_BYTES;
                    const uint32_t b_dst = a_dst + A_BYTES;
                    mbar_arrive_expect_tx(full_bar(stage), STAGE_BYTES);
                    tma_load_2d(a_dst, &tmA, full_bar(stage), kb * BK, arow, pol_act);
                    if (MODE == 0) {
                        tma_load_2d(b_dst, &tmB0, full_bar(stage), kb * BK, brow, pol_w);
                        tma_load_2d(b_dst + B_BYTES / 2, &tmB1, full_bar(stage), kb * BK, brow, pol_w);
                    } else {
                        tma_load_2d(b_dst, &tmB0, full_bar(stage), kb * BK, brow, pol_w);
                    }
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                report(st, kStatusTimeout);
                *abort_flag = 1;
            }
            // Drain: every stage's most recent load must have landed before the CTA exits.
            if (*abort_flag) {
                for (int s = 0; s < STAGES; ++s) {
                    if (issued <= s) continue;
                    const long long last = issued - 1 - ((issued - 1 - s) % STAGES);
                    const uint32_t par = static_cast<uint32_t>((last / STAGES) & 1);
                    mbar_wait(full_bar(s), par, st, nullptr);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc = idesc_bf16_f32(BM, ACC_COLS);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, st, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, st, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = tiles_u32 + stage * STAGE_BYTES;
                    const uint64_t adesc = sdesc_kmajor_sw128(a_addr);
                    const uint64_t bdesc = sdesc_kmajor_sw128(a_addr + A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        // +32 bytes of K per step = +2 in the descriptor's 16-byte address units
                        mma_bf16_ss(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kb | k) != 0);
                    }
                    mma_commit(empty_bar(stage));   // frees this smem stage when the MMAs finish
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(accf_bar(acc));          // accumulator ready for the epilogue
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) {
                report(st, kStatusTimeout);
                *abort_flag = 1;
            }
            // All MMAs issued by this thread must finish before tensor memory is freed.
            mma_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, st, nullptr)) report(st, kStatusTimeout);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;   // the TMEM lane quadrant this warp may read
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            int e, mb, nb;
            tc_decode_tile(prefix, n, p.ntiles, p.group_m, tile, e, mb, nb);
            if (!mbar_wait_warp(accf_bar(acc), acc_phase, st, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const int rloc = mb * BM + q * 32 + lane;      // row inside the expert
            const bool valid = rloc < counts[e];
            const int row = offsets[e] + rloc;
            const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * ACC_COLS) +
                                   (static_cast<uint32_t>(q * 32) << 16);
            int a = 0;
            if (MODE == 0) {
                __nv_bfloat16* hrow = p.H + static_cast<size_t>(valid ? row : 0) * p.ldH + nb * 128;
#pragma unroll 1
                for (int c = 0; c < 128; c += 32) {
                    uint32_t av[32], bv[32];
                    tmem_ld_32x32b_x32(tbase + c, av);
                    tmem_ld_32x32b_x32(tbase + 128 + c, bv);
                    tmem_ld_wait();
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float a0 = __uint_as_float(av[2 * j]), a1 = __uint_as_float(av[2 * j + 1]);
                        const float b0 = __uint_as_float(bv[2 * j]), b1 = __uint_as_float(bv[2 * j + 1]);
                        packed[j] = pack_bf16x2(silu_f(a0) * b0, silu_f(a1) * b1);
                    }
                    if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(hrow + c);
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
                    }
                }
            } else {
                a = valid ? p.perm[row] : 0;
                const float g = valid ? p.topk_w[a] : 0.0f;
                float* yrow = p.Ys + static_cast<size_t>(a) * p.ldY + nb * 256;
#pragma unroll 1
                for (int c = 0; c < 256; c += 32) {
                    uint32_t ov[32];
                    tmem_ld_32x32b_x32(tbase + c, ov);
                    tmem_ld_wait();
                    if (valid) {
                        float4* dst = reinterpret_cast<float4*>(yrow + c);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            dst[v] = make_float4(g * __uint_as_float(ov[4 * v]), g * __uint_as_float(ov[4 * v + 1]),
                                                 g * __uint_as_float(ov[4 * v + 2]), g * __uint_as_float(ov[4 * v + 3]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(acce_bar(acc));
            if (MODE == 1 && p.comb.cnt) {
                combine_arrive(p.comb, p.Ys, p.ldY, valid, a, 2 * nb, lane);
                combine_arrive(p.comb, p.Ys, p.ldY, valid, a, 2 * nb + 1, lane);
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (!ok) {
            if (lane == 0) report(st, kStatusTimeout);
            *abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Row-major bf16 matrix [rows][cols] -> tensor map with a (64 x box_rows) box,
// 128-byte swizzle, zero fill outside the matrix.
bool encode_map_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn || rows == 0 || cols == 0) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major byte matrix [rows][cols] (cols a multiple of 64) -> tensor map
// with a (64-byte x 128-row) box and 64-byte swizzle: 16-byte chunk c of box
// row r lands at chunk c ^ ((r / 2) % 4) of that row.
bool encode_map_u8_sw64(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols) {
    auto fn = encode_fn();
    if (!fn || rows == 0 || cols == 0) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {64, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int MODE>
static cudaError_t launch_tc(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, TcArgs args,
                             int num_sms, cudaStream_t s) {
    // Weights are read by every 128-row block of their expert at about the same
    // time; keeping them at high L2 priority measured ~3% fewer cycles than
    // evict_first on the T=4096 prefill.
    args.w_policy = 2;
    auto kern = tc_grouped_gemm_kernel<MODE>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(SMEM_BYTES));
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(num_sms), dim3(THREADS), SMEM_BYTES, s, a, b0, b1, args);
}

cudaError_t launch_tc_gemm13(const CUtensorMap& mapXp, const CUtensorMap& mapW1, const CUtensorMap& mapW3,
                             const int* sched, int n, int d, int F, int R, __nv_bfloat16* H, KStatus st, int num_sms,
                             cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    if (n > MAX_EXPERTS) return cudaErrorInvalidValue;
    TcArgs args{};
    args.sched = sched;
    args.n = n;
    args.kblocks = d / BK;
    args.ntiles = F / 128;
    args.group_m = tile_group_rows(BM, d);
    args.b_rows_per_e = F;
    args.H = H;
    args.ldH = F;
    args.st = st;
    return launch_tc<0>(mapXp, mapW1, mapW3, args, num_sms, s);
}

cudaError_t launch_tc_gemm2(const CUtensorMap& mapH, const CUtensorMap& mapW2, const int* sched, int n, int d, int F,
                            int R, float* Ys, const int32_t* perm, const float* topk_w, const CombineArgs& comb,
                            KStatus st, int num_sms, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    if (n > MAX_EXPERTS) return cudaErrorInvalidValue;
    TcArgs args{};
    args.sched = sched;
    args.n = n;
    args.kblocks = F / BK;
    args.ntiles = d / 256;
    args.group_m = tile_group_rows(BM, F);
    args.b_rows_per_e = d;
    args.Ys = Ys;
    args.ldY = d;
    args.perm = perm;
    args.topk_w = topk_w;
    args.comb = comb;
    args.st = st;
    return launch_tc<1>(mapH, mapW2, mapW2, args, num_sms, s);
}

}  // namespace moe
