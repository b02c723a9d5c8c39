// gemm_tc2.cu -- the grouped expert GEMMs on CTA pairs (tcgen05 cta_group::2).
//
// Same two products as gemm_tc.cu (aiqianji 3.2.4, code block D):
//
//   MODE 0 (W1/W3 + SwiGLU):  H[r][f] = SiLU(Xp[r] . W1[e][f]) * (Xp[r] . W3[e][f])
//   MODE 1 (W2 + gate):       Ys[a][i] = g_a * (H[r] . W2[e][i]),   a = perm[r]
//
// but each tile is 256 rows of one expert x 256 accumulator columns, computed
// by two CTAs on neighbouring SMs.  CTA r of the pair holds rows
// [128r, 128r+128) of the tile's A operand and rows [128r, 128r+128) of its
// 256-row B operand; one MMA instruction, issued by the even CTA, reads both
// CTAs' shared memory and leaves each CTA's 128 rows x 256 columns of the
// product in that CTA's own tensor memory.  Per k-step a CTA therefore loads
// 16 KB of A and 16 KB of B (32 KB) for the work that costs a single-CTA
// 128 x 256 tile 48 KB, so the operand feed from L2 drops by a third and the
// ring has room for 7 stages.
//
//   MODE 0: CTA 0 loads the 128 W1 rows of the tile's features, CTA 1 the 128
//           W3 rows of the same features: accumulator columns 0-127 are
//           X.W1^T and 128-255 are X.W3^T for every row, as in gemm_tc.cu.
//   MODE 1: CTA r loads W2 rows nb*256 + 128r + [0, 128): columns are the
//           tile's 256 output features in order.
//
// Expert groups are covered by 256-row tiles, except that a group whose last
// tile would hold at most 128 rows ends with a 128-row tile: an M = 128 pair
// MMA, 64 rows from each CTA.  That shape fills all 128 lanes of each CTA's
// tensor memory but only 128 columns: lanes 0-63 hold the 64 rows for output
// columns 0-127 (the even CTA's half of B) and lanes 64-127 hold the same rows
// for columns 128-255 (the odd CTA's half).  So in MODE 0 such a tile loads,
// in CTA r, the W1 rows and then the W3 rows of features [64r, 64r+64) of the
// tile's 128, and every lane again holds both halves of its SwiGLU products.
// Rows past a group's end are computed and dropped in the epilogue.
//
// Roles (6 warps per CTA, both CTAs): warp 0 lane 0 issues the CTA's TMA loads;
// their completion is counted on the even CTA's full barrier (which expects
// both CTAs' bytes).  Warp 1 allocates the pair's tensor memory; in the even
// CTA its lane 0 waits for full stages and issues the MMAs, and its commits
// arrive on both CTAs' empty-stage and accumulator-full barriers.  Warps 2-5
// of each CTA drain their own accumulator rows and tell the even CTA (8
// arrivals per accumulator) that the columns can be reused.  Every wait is
// bounded as in gemm_tc.cu; the pair meets at a cluster barrier before tensor
// memory is freed and before either CTA exits.
#include <cudaTypedefs.h>

#include "combine_epi.cuh"
#include "kernels.h"

namespace moe {

namespace {
constexpr int Q_BK = 64;
constexpr int Q_UMMA_K = 16;
constexpr int Q_STAGES = 7;
constexpr int Q_A_BYTES = 128 * Q_BK * 2;          // this CTA's 128 rows of A
constexpr int Q_B_BYTES = 128 * Q_BK * 2;          // this CTA's 128 rows of B
constexpr int Q_STAGE_BYTES = Q_A_BYTES + Q_B_BYTES;
constexpr int Q_ACC_COLS = 256;
constexpr int Q_TMEM_COLS = 512;
constexpr int Q_THREADS = 192;
constexpr int Q_EPI_WARPS = 4;
constexpr int Q_MAX_EXPERTS = 32;
constexpr int Q_NUM_BARS = 2 * Q_STAGES + 2 + 2 + 1;   // full, empty, acc_full, acc_empty, drain
constexpr size_t Q_SMEM_BYTES = 1024 /*alignment slack*/ + static_cast<size_t>(Q_STAGES) * Q_STAGE_BYTES +
                                Q_NUM_BARS * 8 + 16 + (3 * Q_MAX_EXPERTS + 4) * 4;
constexpr int Q_PAIR_ROWS = 256;
}  // namespace

struct PairArgs {
    const int* sched;
    int n;
    int kblocks;          // K / 64
    int ntiles;           // N blocks per expert
    int group_m;          // 256-row blocks per tile group
    int b_rows_per_e;     // rows of the B tensors per expert (F for MODE 0, d for MODE 1)
    __nv_bfloat16* H;     // MODE 0 output [R][F]
    int ldH;
    float* Ys;            // MODE 1 output [R][d], by flat assignment
    int ldY;
    const int32_t* perm;
    const float* topk_w;
    CombineArgs comb;     // MODE 1: fused combine into y (comb.cnt null: Ys only)
    KStatus st;
};

// tile -> (expert, 256-row block, N block, 128-row tile?); expert-major, then
// groups of group_m row blocks, then N block, then row block (as in gemm_tc.cu).
__device__ __forceinline__ void pair_decode_tile(const int* prefix, const int* counts, int n, int ntiles, int group_m,
                                                 int tile, int& e, int& mb, int& nb, bool& half) {
    int k = 0;
    while (k + 1 < n && prefix[k + 1] * ntiles <= tile) ++k;
    const int mt = prefix[k + 1] - prefix[k];
    const int local = tile - prefix[k] * ntiles;
    const int g = local / (group_m * ntiles);   // row-block groups, as in tc_decode_tile
    const int mg = min(group_m, mt - g * group_m);
    const int r = local - g * group_m * ntiles;
    e = k;
    nb = r / mg;
    mb = g * group_m + r % mg;
    const int rem = counts[k] - mb * Q_PAIR_ROWS;   // rows of the group from this tile on
    half = rem <= 128;
}

template <int MODE>
__global__ void __launch_bounds__(Q_THREADS, 1)
    tc_pair_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB0h,
                        const __grid_constant__ CUtensorMap tmB1h, PairArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t tiles_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t* tiles_ptr = smem_raw + (tiles_u32 - raw_u32);
    uint64_t* bars = reinterpret_cast<uint64_t*>(tiles_ptr + Q_STAGES * Q_STAGE_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Q_NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_sched = reinterpret_cast<int*>(tmem_slot + 4);   // counts [n], offsets [n+1], prefix [n+1]

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (Q_STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * Q_STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * Q_STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * Q_STAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = static_cast<int>(cluster_id_x()), ncl = static_cast<int>(ncluster_x());
    const int n = p.n;
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < Q_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * Q_EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB0);
        if (MODE == 0) {
            tma_prefetch_desc(&tmB1);
            tma_prefetch_desc(&tmB0h);
            tma_prefetch_desc(&tmB1h);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), Q_TMEM_COLS);
        tmem_relinquish_pair();
    }
    // Everything above touches no buffer of the layer; the schedule and the
    // activations come from the kernels before this one.
    griddep_wait();
    for (int i = threadIdx.x; i < 2 * n + 1; i += Q_THREADS) s_sched[i] = p.sched[i];
    __syncthreads();
    if (threadIdx.x == 0) {
        int* prefix = s_sched + 2 * n + 1;
        int acc = 0;
        for (int e = 0; e < n; ++e) {
            prefix[e] = acc;
            acc += (s_sched[e] + Q_PAIR_ROWS - 1) / Q_PAIR_ROWS;
        }
        prefix[n] = acc;
    }
    tc_fence_before();
    __syncthreads();
    // Both CTAs' barriers are initialised before either CTA's TMA or the
    // leader's commits can reach them.
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int* counts = s_sched;
    const int* offsets = s_sched + n;
    const int* prefix = s_sched + 2 * n + 1;
    const int total = prefix[n] * p.ntiles;
    const KStatus st = p.st;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            const uint64_t pol_act = policy_evict_last();
            const uint64_t pol_w = policy_evict_last();
            const CUtensorMap* mapB = (MODE == 0 && rank == 1) ? &tmB1 : &tmB0;
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            // this CTA's A and B rows for a tile
            auto tile_rows = [&](int t, int& ar, int& br, bool& hf) {
                int e2, mb2, nb2;
                pair_decode_tile(prefix, counts, n, p.ntiles, p.group_m, t, e2, mb2, nb2, hf);
                ar = offsets[e2] + mb2 * Q_PAIR_ROWS + static_cast<int>(rank) * (hf ? 64 : 128);
                br = e2 * p.b_rows_per_e +
                     (MODE == 0 ? nb2 * 128 + (hf ? 64 * static_cast<int>(rank) : 0)
                                : nb2 * 256 + static_cast<int>(rank) * 128);
            };
            for (int tile = cid; tile < total && ok; tile += ncl) {
                int arow, brow;
                bool half;
                tile_rows(tile, arow, brow, half);
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1u, st, abort_flag)) { ok = false; break; }
                    const uint32_t a_dst = tiles_u32 + stage * Q_STAGE_BYTES;
                    const uint32_t b_dst = a_dst + Q_A_BYTES;
                    const uint32_t full_leader = mapa_shared(full_bar(stage), 0);
                    if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * Q_STAGE_BYTES);
                    tma_load_2d_pair(a_dst, &tmA, full_leader, kb * Q_BK, arow, pol_act);
                    if (MODE == 0 && half) {
                        // 64 W1 rows then the 64 W3 rows of the same features
                        tma_load_2d_pair(b_dst, &tmB0h, full_leader, kb * Q_BK, brow, pol_w);
                        tma_load_2d_pair(b_dst + Q_B_BYTES / 2, &tmB1h, full_leader, kb * Q_BK, brow, pol_w);
                    } else {
                        tma_load_2d_pair(b_dst, mapB, full_leader, kb * Q_BK, brow, pol_w);
                    }
                    ++issued;
                    if (++stage == Q_STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                report(st, kStatusTimeout);
                *abort_flag = 1;
            }
            if (*abort_flag && issued > 0) {
                // The loads count on the even CTA's barriers, which may never
                // complete once the pair has given up; give the copies already
                // issued (16 KB each, served in microseconds) 50 us to land
                // before shared memory can be released.
                const uint64_t t0 = globaltimer_ns();
                while (globaltimer_ns() - t0 < 50000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (rank == 0 && lane == 0) {
            // ---------------- MMA issuer (even CTA only) ----------------
            constexpr uint32_t idesc_full = idesc_bf16_f32(2 * 128, Q_ACC_COLS);
            constexpr uint32_t idesc_half = idesc_bf16_f32(2 * 64, Q_ACC_COLS);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int tile = cid; tile < total && ok; tile += ncl) {
                int e, mb, nb;
                bool half;
                pair_decode_tile(prefix, counts, n, p.ntiles, p.group_m, tile, e, mb, nb, half);
                const uint32_t idesc = half ? idesc_half : idesc_full;
                if (!mbar_wait_cluster(acce_bar(acc), acc_phase ^ 1u, st, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Q_ACC_COLS);
                for (int kb = 0; kb < p.kblocks; ++kb) {
                    if (!mbar_wait_cluster(full_bar(stage), phase, st, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = tiles_u32 + stage * Q_STAGE_BYTES;
                    const uint64_t adesc = sdesc_kmajor_sw128(a_addr);
                    const uint64_t bdesc = sdesc_kmajor_sw128(a_addr + Q_A_BYTES);
#pragma unroll
                    for (int k = 0; k < Q_BK / Q_UMMA_K; ++k)
                        mma_bf16_ss_pair(d_tmem, adesc + 2u * k, bdesc + 2u * k, idesc, (kb | k) != 0);
                    mma_commit_pair_mc(empty_bar(stage), 0x3);   // frees the stage in both CTAs
                    if (++stage == Q_STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair_mc(accf_bar(acc), 0x3);          // both CTAs' accumulator rows ready
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) {
                report(st, kStatusTimeout);
                *abort_flag = 1;
            }
            // Every MMA issued must finish before the pair frees tensor memory.
            mma_commit_pair_mc(drain_bar, 0x1);
            if (!mbar_wait_cluster(drain_bar, 0, st, nullptr)) report(st, kStatusTimeout);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..5 of both CTAs) ----------------
        const int q = warp & 3;   // the TMEM lane quadrant this warp may read
        const uint32_t acce_leader0 = mapa_shared(acce_bar(0), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int tile = cid; tile < total; tile += ncl) {
            int e, mb, nb;
            bool half;
            pair_decode_tile(prefix, counts, n, p.ntiles, p.group_m, tile, e, mb, nb, half);
            if (!mbar_wait_cluster_warp(accf_bar(acc), acc_phase, st, abort_flag)) { ok = false; break; }
            tc_fence_after();
            // Full tile: lane L of this CTA's tensor memory is tile row 128*rank + L,
            // all 256 columns.  128-row tile: lane L is tile row 64*rank + (L % 64),
            // and holds output columns [128*(L / 64), +128) in tensor-memory
            // columns 0..127.
            const int hcol = half ? (q >> 1) : 0;
            const int rloc = mb * Q_PAIR_ROWS +
                             (half ? static_cast<int>(rank) * 64 + (q & 1) * 32 + lane
                                   : static_cast<int>(rank) * 128 + q * 32 + lane);   // row in the expert
            const bool valid = rloc < counts[e];
            const int row = offsets[e] + rloc;
            const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * Q_ACC_COLS) +
                                   (static_cast<uint32_t>(q * 32) << 16);
            int a = 0;
            if (MODE == 0) {
                // features of this thread: full tile nb*128 + [0,128) with W3 at column
                // offset 128; 128-row tile nb*128 + 64*hcol + [0,64) with W3 at offset 64
                const int nfeat = half ? 64 : 128;
                __nv_bfloat16* hrow = p.H + static_cast<size_t>(valid ? row : 0) * p.ldH + nb * 128 + 64 * hcol;
#pragma unroll 1
                for (int c = 0; c < nfeat; c += 32) {
                    uint32_t av[32], bv[32];
                    tmem_ld_32x32b_x32(tbase + c, av);
                    tmem_ld_32x32b_x32(tbase + nfeat + c, bv);
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
                const int nout = half ? 128 : 256;
                float* yrow = p.Ys + static_cast<size_t>(a) * p.ldY + nb * 256 + 128 * hcol;
#pragma unroll 1
                for (int c = 0; c < nout; c += 32) {
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
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(acce_leader0 + 8u * acc);
            if (MODE == 1 && p.comb.cnt) {
                if (half) {
                    combine_arrive(p.comb, p.Ys, p.ldY, valid, a, 2 * nb + hcol, lane);
                } else {
                    combine_arrive(p.comb, p.Ys, p.ldY, valid, a, 2 * nb, lane);
                    combine_arrive(p.comb, p.Ys, p.ldY, valid, a, 2 * nb + 1, lane);
                }
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
    // Neither CTA frees tensor memory or exits while the other may still use it
    // (the leader's MMAs write the odd CTA's tensor memory and read its
    // shared memory; the odd CTA arrives on the leader's barriers).
    cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Q_TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side

namespace {
// Clusters of two that can be resident at once with one CTA per SM (0 if the
// query fails).  Cached per kernel.
template <int MODE>
int pair_clusters(int num_sms) {
    static int cached = -1;
    if (cached >= 0) return cached;
    auto kern = tc_pair_gemm_kernel<MODE>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Q_SMEM_BYTES)) !=
        cudaSuccess) {
        cudaGetLastError();
        cached = 0;
        return cached;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms & ~1);
    cfg.blockDim = dim3(Q_THREADS);
    cfg.dynamicSmemBytes = Q_SMEM_BYTES;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        nc = 0;
    }
    if (nc > num_sms / 2) nc = num_sms / 2;
    cached = nc;
    return cached;
}

template <int MODE>
cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1, const CUtensorMap& b0h,
                        const CUtensorMap& b1h, PairArgs args, int num_sms, cudaStream_t s) {
    const int nc = pair_clusters<MODE>(num_sms);
    if (nc <= 0) return cudaErrorNotSupported;
    auto kern = tc_pair_gemm_kernel<MODE>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * nc);
    cfg.blockDim = dim3(Q_THREADS);
    cfg.dynamicSmemBytes = Q_SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a, b0, b1, b0h, b1h, args);
}
}  // namespace

bool pair_gemm_available(int num_sms) { return pair_clusters<0>(num_sms) > 0 && pair_clusters<1>(num_sms) > 0; }

cudaError_t launch_pair_gemm13(const CUtensorMap& mapXp, const CUtensorMap& mapW1, const CUtensorMap& mapW3,
                               const CUtensorMap& mapW1_64, const CUtensorMap& mapW3_64, const int* sched, int n,
                               int d, int F, int R, __nv_bfloat16* H, KStatus st, int num_sms, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    if (n > Q_MAX_EXPERTS) return cudaErrorInvalidValue;
    PairArgs args{};
    args.sched = sched;
    args.n = n;
    args.kblocks = d / Q_BK;
    args.ntiles = F / 128;
    args.group_m = tile_group_rows(Q_PAIR_ROWS, d);
    args.b_rows_per_e = F;
    args.H = H;
    args.ldH = F;
    args.st = st;
    return launch_pair<0>(mapXp, mapW1, mapW3, mapW1_64, mapW3_64, args, num_sms, s);
}

cudaError_t launch_pair_gemm2(const CUtensorMap& mapH, const CUtensorMap& mapW2_128, const int* sched, int n, int d,
                              int F, int R, float* Ys, const int32_t* perm, const float* topk_w,
                              const CombineArgs& comb, KStatus st, int num_sms, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    if (n > Q_MAX_EXPERTS) return cudaErrorInvalidValue;
    PairArgs args{};
    args.sched = sched;
    args.n = n;
    args.kblocks = F / Q_BK;
    args.ntiles = d / 256;
    args.group_m = tile_group_rows(Q_PAIR_ROWS, F);
    args.b_rows_per_e = d;
    args.Ys = Ys;
    args.ldY = d;
    args.perm = perm;
    args.topk_w = topk_w;
    args.comb = comb;
    args.st = st;
    return launch_pair<1>(mapH, mapW2_128, mapW2_128, mapW2_128, mapW2_128, args, num_sms, s);
}

}  // namespace moe
