// decode_fused.cu -- the whole MoE layer for small batches in one persistent
// kernel.
//
// A decode-sized batch streams each touched expert's weights once (the
// memory-vs-compute remark of the xyznot summary, "Limitations"), so its time
// is the weights' bytes over HBM bandwidth plus whatever the layer spends
// outside the streaming.  Run as five kernels (routing, W1/W3 streaming,
// SwiGLU, W2 streaming, combine; decode_tc.cu), every kernel boundary costs a
// launch, a pipeline fill and a tail.  Here one cooperative launch with one CTA
// per SM does every step, with grid-wide barriers between the steps that need
// the whole grid's results:
//
//   P0  routing: CTA c routes tokens c, c+G, ... with the routing kernel's
//       small-batch arithmetic (route_fused.cu: sixteen row segments per token,
//       the same fp32 sums in the same order), so the experts chosen here are
//       the ones moe_route reports; with RMSNorm the row's 1/rms is published.
//                                                       -- grid barrier 1
//   P1  dispatch, redundantly in every CTA from the published top-k (counts,
//       exclusive scan, the stable expert-contiguous order); CTA c then
//       gathers (and normalises) rows c, c+G, ... of that order into Xp.
//                                                       -- grid barrier 2
//   P2  W1/W3 weight streaming as tc_decode_kernel<0> (swap-AB tcgen05 MMAs,
//       K split S ways, fp32 partial sums).          -- grid barrier 3
//   P3  SwiGLU of the summed partials into H (bf16), spread over the grid.
//                                                       -- grid barrier 4
//   P4  W2 weight streaming as tc_decode_kernel<1>.   -- grid barrier 5
//   P5  combine: gate, slot sum in slot order, optional residual, one
//       rounding, spread over the grid.
//
// Roles after P1 (6 warps): warp 0 lane 0 issues TMA loads for P2 and then P4
// (the P4 token rows only after barrier 4, which it watches), warp 1 owns
// tensor memory and issues the MMAs of both, warps 2-5 drain accumulators,
// and between the streaming steps run P3 and P5 and the barriers.  Every wait
// is bounded; a wait that runs out raises the CTA's abort flag and records a
// timeout, and the grid's other waits then run out too.  Data written during
// the kernel by other CTAs is read through L2 (ld.cg), never the read-only
// path, and rows that TMA reads are fenced for the async proxy by their
// writers and their readers.
#include "kernels.h"
#include "route_common.cuh"

namespace moe {

namespace {
constexpr int FD_BK = 64;
constexpr int FD_UMMA_K = 16;
constexpr int FD_A_BYTES = 128 * FD_BK * 2;   // one 128-row weight tile, 16 KB
constexpr int FD_B_BOX = 32;                  // token rows per TMA box
constexpr int FD_THREADS = 192;
constexpr int FD_WARPS = FD_THREADS / 32;
constexpr int FD_EPI_THREADS = 128;
constexpr int FD_MAX_EXPERTS = 32;
constexpr int FD_MAX_STAGES = 8;
constexpr int FD_NUM_BARS = 2 * FD_MAX_STAGES + 2 + 2 + 1;
constexpr int FD_TMEM_COLS = 512;
constexpr int FD_VQ = 16;                     // row segments per token of the small-batch router
constexpr int FD_BAR_STRIDE = 64;             // ints between barrier words (separate 128-byte lines)

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// The sum of S K-split partials, added in split order, for data written by
// other CTAs during this kernel (read through L2).
__device__ __forceinline__ float4 sum_splits_cg(const float4* p, size_t stride, int S) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < S; s0 += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (s0 + j < S) v[j] = __ldcg(p + static_cast<size_t>(s0 + j) * stride);
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

// One thread: arrive at a grid barrier and wait until `arrivals` threads have
// arrived (bounded).  Count and generation words as in route_fused.cu; they
// return to their starting state (count 0) after every complete barrier.
__device__ __forceinline__ bool fd_grid_barrier(int* words, int arrivals, const KStatus& st,
                                                const volatile int* abort_flag) {
    int* cnt = words;
    int* gen = words + FD_BAR_STRIDE / 2;
    const int g = ld_acquire_gpu(gen);
    __threadfence();
    const int prev = atomicAdd(cnt, 1);
    if (prev == arrivals - 1) {
        atomicExch(cnt, 0);
        __threadfence();
        st_release_gpu(gen, g + 1);
        return true;
    }
    const uint64_t t0 = globaltimer_ns();
    uint32_t it = 0;
    while (ld_acquire_gpu(gen) == g) {
        if ((++it & 63u) == 0) {
            if (abort_flag && *abort_flag) return false;
            if (globaltimer_ns() - t0 > st.wait_ns) return false;
        }
    }
    return true;
}
}  // namespace

struct FusedDecodeArgs {
    const __nv_bfloat16* x;       // [T][d] tokens (with NORM: the residual rows h)
    const float* Wg;              // [n][d]
    const float* bias;            // [n] or null
    const __nv_bfloat16* resid;   // [T][d] added before the output rounding, or null (may be x)
    __nv_bfloat16* y;             // [T][d] (may be x with NORM: the block updates h in place)
    int T, d, F, n, K;
    float norm_eps;
    int32_t* topk_idx;            // [T*K]
    float* topk_w;                // [T*K]
    float* rstd;                  // [T] (NORM)
    int* sched;                   // counts, offsets, 128-row tile prefix (written by CTA 0)
    int32_t* perm;                // [R] (written by CTA 0)
    int32_t* inv;                 // [R] (written by CTA 0)
    __nv_bfloat16* Xp;            // [R][d] gathered rows
    __nv_bfloat16* H;             // [R][F]
    float* Pa;                    // [S13][R][F]
    float* Pb;
    float* P2;                    // [S2][R][d]
    int* bar;                     // 5 barriers x FD_BAR_STRIDE ints, zero between calls
    int S13, kbs13, S2, kbs2;     // K splits and 64-wide k-blocks per split of the two GEMMs
    int n_max;                    // token columns per item, at most (T rounded up to 32)
    int stages, stage_bytes, acc_stride, acc_sets;
    KStatus st;
};

static size_t fused_smem_bytes(int stages, int stage_bytes, int R) {
    return 1024 + static_cast<size_t>(stages) * stage_bytes + FD_NUM_BARS * 8 + 32 +
           (3 * FD_MAX_EXPERTS + 2) * 4 + FD_MAX_EXPERTS * 4 + static_cast<size_t>(2 * R) * 4 +
           static_cast<size_t>(FD_VQ) * 32 * 4 + FD_VQ * 4;
}

template <int NMAX, bool NORM>
__global__ void __launch_bounds__(FD_THREADS, 1)
    tc_decode_fused_kernel(const __grid_constant__ CUtensorMap tmW1, const __grid_constant__ CUtensorMap tmW3,
                           const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmXp,
                           const __grid_constant__ CUtensorMap tmH, FusedDecodeArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t ring_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t* ring_ptr = smem_raw + (ring_u32 - raw_u32);
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring_ptr + static_cast<size_t>(p.stages) * p.stage_bytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + FD_NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_flag = reinterpret_cast<int*>(tmem_slot + 2);
    int* s_sched = reinterpret_cast<int*>(tmem_slot + 8);           // counts [n], offsets [n+1], prefix [n+1]
    int* s_touched = s_sched + 3 * FD_MAX_EXPERTS + 2;               // touched experts; count in the last slot
    const int R = p.K * p.T;
    int* s_perm = s_touched + FD_MAX_EXPERTS;                        // [R]
    int* s_inv = s_perm + R;                                         // [R]
    float* s_red = reinterpret_cast<float*>(s_inv + R);              // [FD_VQ][32] router segment sums
    float* s_ss = s_red + FD_VQ * 32;                                // [FD_VQ] sums of squares

    const uint32_t bar0 = smem_u32(bars);
    const int NS = p.stages;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (FD_MAX_STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * FD_MAX_STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * FD_MAX_STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * FD_MAX_STAGES + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int n = p.n, d = p.d, F = p.F, K = p.K, T = p.T;
    const KStatus st = p.st;
    auto barrier_words = [&](int i) { return p.bar + i * FD_BAR_STRIDE; };

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), FD_EPI_THREADS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW1);
        tma_prefetch_desc(&tmW3);
        tma_prefetch_desc(&tmW2);
        tma_prefetch_desc(&tmXp);
        tma_prefetch_desc(&tmH);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), FD_TMEM_COLS);
        tmem_relinquish();
    }
    // The generation of barrier 4 before anyone can pass it in this call: the
    // TMA producer waits for it to move before loading SwiGLU rows.
    const int h_gen0 = ld_acquire_gpu(barrier_words(3) + FD_BAR_STRIDE / 2);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // One thread meets the grid at barrier i; the rest of the CTA waits for it.
    auto grid_sync_all = [&](int i) -> bool {
        __threadfence();   // this thread's writes before the CTA's arrival
        __syncthreads();
        if (tid == 0) *s_flag = fd_grid_barrier(barrier_words(i), G, st, abort_flag) ? 1 : 0;
        __syncthreads();
        return *s_flag != 0;
    };

    bool ok = true;
    // ---------------- P0: routing (the small-batch router's arithmetic) ----------------
    for (int t = b; t < T && ok; t += G) {
        const __nv_bfloat16* row = p.x + static_cast<size_t>(t) * d;
        float rs = 1.0f;
        if constexpr (NORM) {
            for (int q = warp; q < FD_VQ; q += FD_WARPS) {
                float ss = 0.0f;
                for (int sg = q; sg * 256 < d; sg += FD_VQ) {
                    const int j0 = sg * 256 + 4 * lane;
                    Raw4<__nv_bfloat16> r0, r1;
                    load_raw4(row, j0, j0 < d, r0);
                    load_raw4(row, j0 + 128, j0 + 128 < d, r1);
                    float u[8];
                    unpack_raw4(r0, &u[0]);
                    unpack_raw4(r1, &u[4]);
#pragma unroll
                    for (int k = 0; k < 8; ++k) ss = fmaf(u[k], u[k], ss);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (lane == 0) s_ss[q] = ss;
            }
            __syncthreads();
            float tot = 0.0f;
#pragma unroll
            for (int qq = 0; qq < FD_VQ; ++qq) tot += s_ss[qq];
            rs = 1.0f / sqrtf(tot / static_cast<float>(d) + p.norm_eps);
            if (tid == 0) p.rstd[t] = rs;
        }
        for (int q = warp; q < FD_VQ; q += FD_WARPS) {
            float acc[NMAX];
#pragma unroll
            for (int e = 0; e < NMAX; ++e) acc[e] = 0.0f;
            for (int sg = q; sg * 256 < d; sg += FD_VQ) {
                const int j0 = sg * 256 + 4 * lane, j1 = j0 + 128;
                const bool h0 = j0 < d, h1 = j1 < d;
                Raw4<__nv_bfloat16> r0, r1;
                load_raw4(row, j0, h0, r0);
                load_raw4(row, j1, h1, r1);
                float xv[8];
                unpack_raw4(r0, &xv[0]);
                unpack_raw4(r1, &xv[4]);
                if constexpr (NORM) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) xv[k] = scale_round<__nv_bfloat16>(xv[k], rs);
                }
#pragma unroll
                for (int e = 0; e < NMAX; ++e) {
                    if (e < n) {
                        const float* w = p.Wg + static_cast<size_t>(e) * d;
                        float4 w0 = make_float4(0.f, 0.f, 0.f, 0.f), w1 = w0;
                        if (h0) w0 = __ldg(reinterpret_cast<const float4*>(w + j0));
                        if (h1) w1 = __ldg(reinterpret_cast<const float4*>(w + j1));
                        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                        float a = acc[e];
#pragma unroll
                        for (int u = 0; u < 8; ++u) a = fmaf(xv[u], wv[u], a);
                        acc[e] = a;
                    }
                }
            }
            lane_transpose_sum<NMAX>(acc, lane);
            constexpr int VF = NMAX >= 32 ? NMAX / 32 : 1;
#pragma unroll
            for (int i = 0; i < VF; ++i) s_red[q * 32 + fr_index<NMAX>(lane, i)] = acc[i];
        }
        __syncthreads();
        if (warp == 0) {
            float l[NMAX];
#pragma unroll
            for (int e = 0; e < NMAX; ++e) {
                float s = 0.0f;
                if (e < n) {
#pragma unroll
                    for (int qq = 0; qq < FD_VQ; ++qq) s += s_red[qq * 32 + e];
                    if (p.bias) s += __ldg(p.bias + e);
                }
                l[e] = s;
            }
            topk_gate_write<NMAX>(l, n, K, t, lane, p.topk_idx, p.topk_w, nullptr, nullptr);
        }
        __syncthreads();
    }
    ok = grid_sync_all(0);

    // ---------------- P1: dispatch (every CTA) and row gather ----------------
    if (ok) {
        if (warp == 0) {
            if (lane < FD_MAX_EXPERTS) s_sched[lane] = 0;
            __syncwarp();
            const unsigned lt = (1u << lane) - 1u;
            for (int pass = 0; pass < 2; ++pass) {
                for (int a0 = 0; a0 < R; a0 += 32) {
                    const int a = a0 + lane;
                    int e = a < R ? __ldcg(p.topk_idx + a) : -1;
                    if (a < R && (e < 0 || e >= n)) {
                        report(st, kStatusBounds);
                        e = -1;
                    }
                    const unsigned same = __match_any_sync(0xffffffffu, e);
                    const int rank = __popc(same & lt);
                    if (pass == 0) {
                        if (e >= 0 && rank == 0) s_sched[e] += __popc(same);
                    } else if (e >= 0) {
                        const int pos = s_sched[n + e] + s_sched[2 * n + 1 + e] + rank;   // offset + placed so far
                        s_perm[pos] = a;
                        s_inv[a] = pos;
                    }
                    __syncwarp();
                    if (pass == 1 && e >= 0 && rank == 0) s_sched[2 * n + 1 + e] += __popc(same);
                    __syncwarp();
                }
                if (pass == 0 && lane == 0) {
                    int run = 0, nt = 0;
                    for (int e = 0; e < n; ++e) {
                        s_sched[n + e] = run;
                        s_sched[2 * n + 1 + e] = 0;   // running placement count during pass 1
                        run += s_sched[e];
                        if (s_sched[e] > 0) s_touched[nt++] = e;
                    }
                    s_sched[2 * n] = run;
                    s_touched[FD_MAX_EXPERTS - 1] = nt;
                }
                __syncwarp();
            }
            // the 128-row tile prefix (the dispatch kernel's schedule layout)
            if (lane == 0) {
                int tp = 0;
                for (int e = 0; e < n; ++e) {
                    s_sched[2 * n + 1 + e] = tp;
                    tp += (s_sched[e] + kTileM - 1) / kTileM;
                }
                s_sched[3 * n + 1] = tp;
            }
        }
        __syncthreads();
        if (b == 0) {
            for (int i = tid; i < 3 * n + 2; i += FD_THREADS) p.sched[i] = s_sched[i];
            for (int i = tid; i < R; i += FD_THREADS) {
                p.perm[i] = s_perm[i];
                p.inv[i] = s_inv[i];
            }
        }
        // rows b, b+G, ... of the expert-contiguous order
        const int rv = d / 8;
        for (int r = b; r < R; r += G) {
            const int t = s_perm[r] / K;
            const uint4* src = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * d);
            uint4* dst = reinterpret_cast<uint4*>(p.Xp + static_cast<size_t>(r) * d);
            float rsv = 1.0f;
            if constexpr (NORM) rsv = __ldcg(p.rstd + t);
            for (int v = tid; v < rv; v += FD_THREADS) {
                uint4 u = __ldg(src + v);
                if constexpr (NORM) u = scale_row_vec<__nv_bfloat16>(u, rsv);
                dst[v] = u;
            }
        }
        fence_proxy_async_global();   // the gathered rows are read by TMA
        ok = grid_sync_all(1);
    }
    if (!ok) {
        if (tid == 0) report(st, kStatusTimeout);
        if (tid == 0) *abort_flag = 1;
    }
    __syncthreads();

    const int* counts = s_sched;
    const int* offsets = s_sched + n;
    const int n_touched = s_touched[FD_MAX_EXPERTS - 1];
    const int items13 = ok ? n_touched * (F / 128) * p.S13 : 0;
    const int items2 = ok ? n_touched * (d / 128) * p.S2 : 0;
    auto item_n = [&](int e) { return max(FD_B_BOX, (counts[e] + FD_B_BOX - 1) / FD_B_BOX * FD_B_BOX); };
    // item -> (expert, weight row block, K split); K split fastest
    auto decode_item = [&](int it, int rblocks, int S, int& e, int& rb, int& sp) {
        sp = it % S;
        const int r = it / S;
        rb = r % rblocks;
        e = s_touched[r / rblocks];
    };

    if (warp == 0) {
        if (lane == 0 && ok) {
            // ---------------- TMA producer: W1/W3, then W2 ----------------
            const uint64_t pol_w = policy_evict_first();   // each weight byte is read once
            const uint64_t pol_x = policy_evict_last();    // token rows are re-read by every row block
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool pok = true;
            for (int ph = 0; ph < 2 && pok; ++ph) {
                const int items = ph == 0 ? items13 : items2;
                const int rblocks = ph == 0 ? F / 128 : d / 128;
                const int S = ph == 0 ? p.S13 : p.S2, kbs = ph == 0 ? p.kbs13 : p.kbs2;
                const int rows_per_e = ph == 0 ? F : d;
                const int a_tiles = ph == 0 ? 2 : 1;
                if (ph == 1) {
                    // the SwiGLU rows exist once the whole grid has passed barrier 4
                    const uint64_t t0 = globaltimer_ns();
                    uint32_t it = 0;
                    while (ld_acquire_gpu(barrier_words(3) + FD_BAR_STRIDE / 2) == h_gen0) {
                        if ((++it & 63u) == 0 && (*abort_flag || globaltimer_ns() - t0 > st.wait_ns)) {
                            pok = false;
                            break;
                        }
                    }
                    if (!pok) break;
                    fence_proxy_async_global();
                }
                for (int it = b; it < items && pok; it += G) {
                    int e, rb, sp;
                    decode_item(it, rblocks, S, e, rb, sp);
                    const int nbox = item_n(e) / FD_B_BOX;
                    const int arow = e * rows_per_e + rb * 128;
                    const int brow = offsets[e];
                    const uint32_t bytes = a_tiles * FD_A_BYTES + nbox * FD_B_BOX * FD_BK * 2;
                    for (int kb = sp * kbs; kb < (sp + 1) * kbs; ++kb) {
                        if (!mbar_wait(empty_bar(stage), phase ^ 1u, st, abort_flag)) { pok = false; break; }
                        const uint32_t a_dst = ring_u32 + stage * p.stage_bytes;
                        const uint32_t b_dst = a_dst + a_tiles * FD_A_BYTES;
                        mbar_arrive_expect_tx(full_bar(stage), bytes);
                        if (ph == 0) {
                            tma_load_2d(a_dst, &tmW1, full_bar(stage), kb * FD_BK, arow, pol_w);
                            tma_load_2d(a_dst + FD_A_BYTES, &tmW3, full_bar(stage), kb * FD_BK, arow, pol_w);
                        } else {
                            tma_load_2d(a_dst, &tmW2, full_bar(stage), kb * FD_BK, arow, pol_w);
                        }
                        const CUtensorMap* tb = ph == 0 ? &tmXp : &tmH;
                        for (int bb = 0; bb < nbox; ++bb)
                            tma_load_2d(b_dst + bb * FD_B_BOX * FD_BK * 2, tb, full_bar(stage), kb * FD_BK,
                                        brow + bb * FD_B_BOX, pol_x);
                        ++issued;
                        if (++stage == NS) { stage = 0; phase ^= 1u; }
                    }
                }
            }
            if (!pok) {
                report(st, kStatusTimeout);
                *abort_flag = 1;
            }
            if (*abort_flag) {
                // every stage's most recent load must land before the CTA exits
                for (int s = 0; s < NS; ++s) {
                    if (issued <= s) continue;
                    const long long last = issued - 1 - ((issued - 1 - s) % NS);
                    mbar_wait(full_bar(s), static_cast<uint32_t>((last / NS) & 1), st, nullptr);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && ok) {
            // ---------------- MMA issuer: W1/W3 items, then W2 items ----------------
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool mok = true;
            for (int ph = 0; ph < 2 && mok; ++ph) {
                const int items = ph == 0 ? items13 : items2;
                const int rblocks = ph == 0 ? F / 128 : d / 128;
                const int S = ph == 0 ? p.S13 : p.S2, kbs = ph == 0 ? p.kbs13 : p.kbs2;
                const int a_tiles = ph == 0 ? 2 : 1;
                for (int it = b; it < items && mok; it += G) {
                    int e, rb, sp;
                    decode_item(it, rblocks, S, e, rb, sp);
                    const uint32_t idesc = idesc_bf16_f32(128, item_n(e));
                    if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, st, abort_flag)) { mok = false; break; }
                    tc_fence_after();
                    const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * p.acc_stride);
                    const uint32_t d1 = d0 + static_cast<uint32_t>(p.n_max);
                    for (int k = 0; k < kbs; ++k) {
                        if (!mbar_wait(full_bar(stage), phase, st, abort_flag)) { mok = false; break; }
                        tc_fence_after();
                        const uint32_t a_addr = ring_u32 + stage * p.stage_bytes;
                        const uint64_t adesc0 = sdesc_kmajor_sw128(a_addr);
                        const uint64_t adesc1 = sdesc_kmajor_sw128(a_addr + FD_A_BYTES);
                        const uint64_t bdesc = sdesc_kmajor_sw128(a_addr + a_tiles * FD_A_BYTES);
#pragma unroll
                        for (int kk = 0; kk < FD_BK / FD_UMMA_K; ++kk) {
                            const uint32_t accum = (k | kk) != 0;
                            mma_bf16_ss(d0, adesc0 + 2u * kk, bdesc + 2u * kk, idesc, accum);
                            if (a_tiles == 2) mma_bf16_ss(d1, adesc1 + 2u * kk, bdesc + 2u * kk, idesc, accum);
                        }
                        mma_commit(empty_bar(stage));
                        if (++stage == NS) { stage = 0; phase ^= 1u; }
                    }
                    if (!mok) break;
                    mma_commit(accf_bar(acc));
                    if (++acc == p.acc_sets) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                }
            }
            if (!mok) {
                report(st, kStatusTimeout);
                *abort_flag = 1;
            }
            mma_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, st, nullptr)) report(st, kStatusTimeout);
        }
        __syncwarp();
    } else if (ok) {
        // ---------------- epilogue warps: partial sums, SwiGLU, combine ----------------
        const int q = warp & 3;
        const int etid = tid - 64;   // 0..127 over the epilogue warps
        int acc = 0;
        uint32_t acc_phase = 0;
        bool eok = true;
        // Each epilogue warp meets the grid on its own (4 G arrivals), so that a warp
        // whose wait ran out cannot leave the others blocked in a CTA barrier.
        auto epi_grid_sync = [&](int i) -> bool {
            __threadfence();   // this lane's writes before the warp's arrival
            __syncwarp();
            int r = 1;
            if (lane == 0) r = fd_grid_barrier(barrier_words(i), 4 * G, st, abort_flag) ? 1 : 0;
            r = __shfl_sync(0xffffffffu, r, 0);
            __syncwarp();
            return r != 0;
        };
        for (int ph = 0; ph < 2 && eok; ++ph) {
            const int items = ph == 0 ? items13 : items2;
            const int rblocks = ph == 0 ? F / 128 : d / 128;
            const int S = ph == 0 ? p.S13 : p.S2;
            const int parts = ph == 0 ? 2 : 1;
            const int ld = ph == 0 ? F : d;
            for (int it = b; it < items; it += G) {
                int e, rb, sp;
                decode_item(it, rblocks, S, e, rb, sp);
                const int N = item_n(e);
                const int cnt = counts[e];
                const int off = offsets[e];
                if (!mbar_wait_warp(accf_bar(acc), acc_phase, st, abort_flag)) { eok = false; break; }
                tc_fence_after();
                const int feat = rb * 128 + q * 32 + lane;   // this thread's weight row = output feature
                const uint32_t t0 =
                    tmem_base + static_cast<uint32_t>(acc * p.acc_stride) + (static_cast<uint32_t>(q * 32) << 16);
                for (int part = 0; part < parts; ++part) {
                    float* P = (ph == 1 ? p.P2 : part == 0 ? p.Pa : p.Pb) + static_cast<size_t>(sp) * R * ld;
                    const uint32_t tp = t0 + static_cast<uint32_t>(part * p.n_max);
                    for (int c = 0; c < N; c += 32) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(tp + c, v);
                        tmem_ld_wait();
                        const int jn = min(32, cnt - c);
                        float* dst = P + static_cast<size_t>(off + c) * ld + feat;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < jn) dst[static_cast<size_t>(j) * ld] = __uint_as_float(v[j]);
                    }
                }
                tc_fence_before();
                mbar_arrive(acce_bar(acc));
                if (++acc == p.acc_sets) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!eok) break;
            if (ph == 0) {
                // every W1/W3 partial sum of the grid is written
                if (!epi_grid_sync(2)) { eok = false; break; }
                // P3: H = bf16(SiLU(a) * b) over the summed partials, slice b of the grid
                const size_t part4 = static_cast<size_t>(R) * F / 4;
                const float4* pa = reinterpret_cast<const float4*>(p.Pa);
                const float4* pb = reinterpret_cast<const float4*>(p.Pb);
                uint2* h2 = reinterpret_cast<uint2*>(p.H);
                for (size_t i = static_cast<size_t>(b) * FD_EPI_THREADS + etid; i < part4;
                     i += static_cast<size_t>(G) * FD_EPI_THREADS) {
                    const float4 a = sum_splits_cg(pa + i, part4, p.S13), bb = sum_splits_cg(pb + i, part4, p.S13);
                    uint2 o;
                    o.x = pack_bf16x2(silu_f(a.x) * bb.x, silu_f(a.y) * bb.y);
                    o.y = pack_bf16x2(silu_f(a.z) * bb.z, silu_f(a.w) * bb.w);
                    h2[i] = o;
                }
                fence_proxy_async_global();   // H is read by TMA
                if (!epi_grid_sync(3)) { eok = false; break; }
            }
        }
        if (eok) {
            // every W2 partial sum of the grid is written
            eok = epi_grid_sync(4);
            if (eok) {
                // P5: y[t][i] = (resid +) sum_k g[t][k] * (sum_s P2[s][inv[t K + k]][i]), one rounding
                const int d4 = d / 4;
                const size_t part4 = static_cast<size_t>(R) * d4;
                const float4* P2 = reinterpret_cast<const float4*>(p.P2);
                for (size_t i = static_cast<size_t>(b) * FD_EPI_THREADS + etid; i < static_cast<size_t>(T) * d4;
                     i += static_cast<size_t>(G) * FD_EPI_THREADS) {
                    const size_t t = i / d4, c = i % d4;
                    float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int k = 0; k < K; ++k) {
                        const size_t a = t * K + k;
                        const size_t row = static_cast<size_t>(s_inv[a]);
                        const float g = __ldcg(p.topk_w + a);
                        const float4 v = sum_splits_cg(P2 + row * d4 + c, part4, p.S2);
                        acc4.x += g * v.x; acc4.y += g * v.y; acc4.z += g * v.z; acc4.w += g * v.w;
                    }
                    if (p.resid) {
                        const uint2 hv = *reinterpret_cast<const uint2*>(p.resid + t * d + 4 * c);
                        const __nv_bfloat162 h0 = *reinterpret_cast<const __nv_bfloat162*>(&hv.x);
                        const __nv_bfloat162 h1 = *reinterpret_cast<const __nv_bfloat162*>(&hv.y);
                        acc4.x = __low2float(h0) + acc4.x;
                        acc4.y = __high2float(h0) + acc4.y;
                        acc4.z = __low2float(h1) + acc4.z;
                        acc4.w = __high2float(h1) + acc4.w;
                    }
                    uint2 o;
                    o.x = pack_bf16x2(acc4.x, acc4.y);
                    o.y = pack_bf16x2(acc4.z, acc4.w);
                    *reinterpret_cast<uint2*>(p.y + t * d + 4 * c) = o;
                }
            }
        }
        if (!eok) {
            if (lane == 0) report(st, kStatusTimeout);
            *abort_flag = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, FD_TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side

namespace {
struct FusedPlan {
    FusedDecodeArgs a;
    size_t smem;
};

// The launch parameters of one call (no side effects); false when the shape is
// outside the kernel's limits.
bool fused_plan(const FusedDecodeInput& in, int num_sms, FusedPlan& pl) {
    if (!fused_decode_supported(in.T, in.d, in.F, in.n, in.K, num_sms)) return false;
    FusedDecodeArgs& a = pl.a;
    a = FusedDecodeArgs{};
    a.x = in.x;
    a.Wg = in.Wg;
    a.bias = in.bias;
    a.resid = in.resid;
    a.y = in.y;
    a.T = in.T;
    a.d = in.d;
    a.F = in.F;
    a.n = in.n;
    a.K = in.K;
    a.norm_eps = in.norm_eps;
    a.topk_idx = in.topk_idx;
    a.topk_w = in.topk_w;
    a.rstd = in.rstd;
    a.sched = in.sched;
    a.perm = in.perm;
    a.inv = in.inv;
    a.Xp = in.Xp;
    a.H = in.H;
    a.Pa = in.Pa;
    a.Pb = in.Pb;
    a.P2 = in.P2;
    a.bar = in.bar;
    a.st = in.st;
    const int R = in.K * in.T;
    const int touched = in.n < R ? in.n : R;
    // the same K splits as the five-kernel path, so both give the same partial sums
    a.S13 = decode_pick_splits(touched * (in.F / 128), in.d / FD_BK, num_sms);
    a.kbs13 = in.d / FD_BK / a.S13;
    a.S2 = decode_pick_splits(touched * (in.d / 128), in.F / FD_BK, num_sms);
    a.kbs2 = in.F / FD_BK / a.S2;
    a.n_max = (in.T + FD_B_BOX - 1) / FD_B_BOX * FD_B_BOX;
    // stages sized for the W1/W3 step (two weight tiles and the token rows); the
    // W2 step uses the same ring
    a.stage_bytes = 2 * FD_A_BYTES + a.n_max * FD_BK * 2;
    a.stages = static_cast<int>((200 * 1024) / a.stage_bytes);
    if (a.stages > FD_MAX_STAGES) a.stages = FD_MAX_STAGES;
    if (a.stages < 2) return false;
    a.acc_stride = 2 * a.n_max;
    a.acc_sets = 2 * a.acc_stride <= FD_TMEM_COLS ? 2 : 1;
    if (a.acc_stride > FD_TMEM_COLS) return false;
    pl.smem = fused_smem_bytes(a.stages, a.stage_bytes, R);
    return true;
}

template <int NMAX, bool NORM>
cudaError_t fused_prepare_t(size_t smem, int num_sms) {
    auto kern = tc_decode_fused_kernel<NMAX, NORM>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, FD_THREADS, smem);
    if (err != cudaSuccess) return err;
    return per_sm >= 1 && num_sms >= 1 ? cudaSuccess : cudaErrorNotSupported;
}

template <int NMAX, bool NORM>
cudaError_t fused_launch_t(const CUtensorMap& mW1, const CUtensorMap& mW3, const CUtensorMap& mW2,
                           const CUtensorMap& mXp, const CUtensorMap& mH, const FusedPlan& pl, int grid,
                           cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(FD_THREADS);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every CTA resident: the grid barriers need it
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_decode_fused_kernel<NMAX, NORM>, mW1, mW3, mW2, mXp, mH, pl.a);
}

}  // namespace

int fused_decode_bar_ints() { return 5 * FD_BAR_STRIDE; }

bool fused_decode_supported(int T, int d, int F, int n, int K, int num_sms) {
    // the routing step reproduces the routing kernel's one-token-per-block
    // arithmetic, which that kernel uses while it has a block for every token
    return T >= 1 && T <= kDecodeMaxT && fused_route_blocks(T, num_sms) == T && K * T <= 512 &&
           n <= FD_MAX_EXPERTS - 1 && d % 256 == 0 && F % 128 == 0;
}

cudaError_t prepare_decode_fused(const FusedDecodeInput& in, int num_sms) {
    FusedPlan pl;
    if (!fused_plan(in, num_sms, pl)) return cudaErrorNotSupported;
    const bool norm = in.rstd != nullptr;
    if (in.n <= 8) return norm ? fused_prepare_t<8, true>(pl.smem, num_sms) : fused_prepare_t<8, false>(pl.smem, num_sms);
    if (in.n <= 16)
        return norm ? fused_prepare_t<16, true>(pl.smem, num_sms) : fused_prepare_t<16, false>(pl.smem, num_sms);
    return norm ? fused_prepare_t<32, true>(pl.smem, num_sms) : fused_prepare_t<32, false>(pl.smem, num_sms);
}

cudaError_t launch_decode_fused(const CUtensorMap& mW1, const CUtensorMap& mW3, const CUtensorMap& mW2,
                                const CUtensorMap& mXp32, const CUtensorMap& mH32, const FusedDecodeInput& in,
                                int num_sms, cudaStream_t s) {
    FusedPlan pl;
    if (!fused_plan(in, num_sms, pl)) return cudaErrorNotSupported;
    const bool norm = in.rstd != nullptr;
    if (in.n <= 8)
        return norm ? fused_launch_t<8, true>(mW1, mW3, mW2, mXp32, mH32, pl, num_sms, s)
                    : fused_launch_t<8, false>(mW1, mW3, mW2, mXp32, mH32, pl, num_sms, s);
    if (in.n <= 16)
        return norm ? fused_launch_t<16, true>(mW1, mW3, mW2, mXp32, mH32, pl, num_sms, s)
                    : fused_launch_t<16, false>(mW1, mW3, mW2, mXp32, mH32, pl, num_sms, s);
    return norm ? fused_launch_t<32, true>(mW1, mW3, mW2, mXp32, mH32, pl, num_sms, s)
                : fused_launch_t<32, false>(mW1, mW3, mW2, mXp32, mH32, pl, num_sms, s);
}

}  // namespace moe
