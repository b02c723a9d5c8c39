// route_fused.cu -- router, dispatch and row gather of the MoE layer in one
// kernel.
//
// What it computes is exactly what the separate router, dispatch and gather
// kernels of route.cu compute (the pages' gate and the one_hot/where walk with
// its hidden_states[top_x] gather, aiqianji 2.1.1 and 3.1.2, code blocks B/C),
// organised so that no step runs on a single block:
//
//   phase 1  every block routes one contiguous range of tokens: fp32 logits
//            x . W_g^T (+ bias) with W_g staged in shared memory, top-k and the
//            softmax over the kept logits, plus the block's per-expert counts;
//   barrier  the blocks publish their counts and meet at one grid-wide
//            barrier (all blocks are resident: one per SM at most);
//   phase 2  every block reads all blocks' counts, so it knows the expert
//            offsets and how many rows of each expert the blocks before it own;
//            it places its own assignments a = t*K + slot at
//            offsets[e] + (rows of e in earlier blocks) + (rank among its own
//            rows of e, in a order) -- the stable expert-contiguous order -- and
//            copies their token rows into Xp.
//
// Block b's tokens precede block b+1's, so the order is the same as a single
// pass over all assignments would give.  Nothing depends on timing: counts are
// order-free sums and every position follows from them.
//
// Logits: block of 16 warps = 4 token groups x 4 warps that split the row;
// warp (g, q) takes the 256-element segments q, q+4, q+8, ... of the row, and
// in each segment lane l takes elements [4l, 4l+4) and [128+4l, 128+4l+4), so
// a warp's float4 reads of W_g cover 512 contiguous bytes (no shared-memory
// bank conflicts) and its x reads are coalesced.  A lane accumulates in
// segment order, the 32 lanes are added by a fixed transpose-and-add pattern,
// and the 4 quarter sums are added in q order before the bias.  The same
// arithmetic serves moe_route, moe_router_logits and moe_forward.
//
// Optional RMSNorm of the rows (the residual blocks of a stack,
// h <- h + MoE(RMSNorm(h))): with NORM the kernel first sums each row's squares
// (fp32, in the same fixed lane/segment/quarter order), takes
// rstd = 1 / sqrt(mean + eps), and every later use of the row -- the router's
// dot products and the gathered expert rows -- sees x = h * rstd rounded to the
// element type, so router and experts get the same values.
//
// The grid barrier: a count and a generation word in the context workspace.
// Each block reads the generation, adds 1 to the count; the last arrival
// resets the count to 0 and advances the generation, the others wait for it
// to advance (bounded; on expiry the block records a timeout and leaves).  The
// words return to their starting state after every complete call, so a CUDA
// graph can replay the launch.  Dependent kernels are released only after
// every block has passed the barrier, so the next call's blocks can never
// meet this call's.
#include "kernels.h"
#include "route_common.cuh"

namespace moe {

namespace {
constexpr int FR_THREADS = 512;
constexpr int FR_WARPS = 16;
constexpr int FR_DS_LARGE = 4;              // warps that split one row (batches of many tokens)
constexpr int FR_ROUND = FR_THREADS;        // assignments placed per round in phase 2

}  // namespace

struct FusedRouteArgs {
    const void* x;
    const float* Wg;
    const float* bias;
    int T, d, n, K;
    int chunk;              // tokens per block (the last block may have fewer)
    int32_t* topk_idx;      // [T*K]
    float* topk_w;          // [T*K]
    float* logits;          // optional [T][n]
    int* sched;             // counts, offsets, 128-row tile prefix
    int32_t* perm;          // [T*K]
    int32_t* inv;           // [T*K]
    void* Xp;               // optional [T*K][d]: gathered rows
    int row_vecs;           // 16-byte vectors per row of x
    int* xchg;              // [0] count, [1] generation, [2 + 32*b + e] block counts
    size_t red_off;         // byte offset of the lane-sum buffer in dynamic shared memory
    float norm_eps;         // NORM: RMSNorm epsilon
    float* rstd;            // NORM: [T] 1 / rms of each row, for the gather
    KStatus st;
};

// SMALL (one token per block, small batches): all 16 warps split the row and
// W_g is read from L2 instead of being staged in shared memory first, which
// would cost more latency than the one token's dot products.
template <typename TX, int NMAX, int TOKW, bool NORM, bool SMALL>
__global__ void __launch_bounds__(FR_THREADS, 1) route_fused_kernel(FusedRouteArgs p) {
    constexpr int FR_DS = SMALL ? FR_WARPS : FR_DS_LARGE;   // warps that split one row
    constexpr int FR_TG = FR_WARPS / FR_DS;                 // token groups per block
    extern __shared__ __align__(16) unsigned char fr_smem[];
    const float* wg_s = SMALL ? p.Wg : reinterpret_cast<const float*>(fr_smem);
    float* red = reinterpret_cast<float*>(fr_smem + p.red_off);   // [FR_DS][TPB][NMAX]
    __shared__ int s_hist[32], s_cnt[32], s_pre[32], s_base[32], s_run[32];
    __shared__ int wtab[FR_WARPS][33];
    __shared__ int s_ok;
    __shared__ float s_ss[FR_TG * TOKW][FR_DS];   // NORM: quarter sums of squares
    __shared__ int s_topk[32];                    // SMALL: the block's token's K experts, in rank order
    constexpr int TPB = FR_TG * TOKW;   // tokens per block iteration
    constexpr int V = TOKW * NMAX;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = p.n, d = p.d, K = p.K;
    const int b = blockIdx.x, G = gridDim.x;

    // W_g is written by no kernel of the layer: stage it before waiting on the
    // previous kernel.
    if (!SMALL) {
        const int total4 = n * d / 4;
        const float4* src = reinterpret_cast<const float4*>(p.Wg);
        float4* dst = reinterpret_cast<float4*>(fr_smem);
        for (int i0 = tid; i0 < total4; i0 += 8 * FR_THREADS) {
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * FR_THREADS;
                v[u] = i < total4 ? __ldg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int i = i0 + u * FR_THREADS;
                if (i < total4) dst[i] = v[u];
            }
        }
    }
    // SMALL: W_g is read from L2 in the loop below; with up to 8 experts this
    // warp's first segment of it is loaded here, before the wait, so that only
    // x's loads follow it (64 registers; more experts would spill).
    constexpr bool WPRE = SMALL && NMAX <= 8;
    float4 wpre[WPRE ? NMAX : 1][2];
    if constexpr (WPRE) {
        const int j0 = (warp % FR_DS) * 256 + 4 * lane, j1 = j0 + 128;
#pragma unroll
        for (int e = 0; e < NMAX; ++e) {
            wpre[e][0] = wpre[e][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (e < p.n) {
                if (j0 < p.d) wpre[e][0] = __ldg(reinterpret_cast<const float4*>(p.Wg + static_cast<size_t>(e) * p.d + j0));
                if (j1 < p.d) wpre[e][1] = __ldg(reinterpret_cast<const float4*>(p.Wg + static_cast<size_t>(e) * p.d + j1));
            }
        }
    }
    if (tid < 32) s_hist[tid] = 0;
    griddep_wait();
    // the previous call has finished: its schedule-ready word goes back to 0
    if (b == 0 && tid == 0) p.xchg[kReadyWord] = 0;
    __syncthreads();

    // ---------------- phase 1: logits, top-k, gates, block counts ----------------
    const int t_begin = b * p.chunk;
    const int t_end = min(p.T, t_begin + p.chunk);
    const TX* x = static_cast<const TX*>(p.x);
    const int tg = warp / FR_DS, q = warp % FR_DS;
    float rs_small = 1.0f;   // SMALL + NORM: the block's token's 1/rms, for the gather
    for (int tb = t_begin; tb < t_end; tb += TPB) {
        float acc[TOKW][NMAX];
#pragma unroll
        for (int j = 0; j < TOKW; ++j)
#pragma unroll
            for (int e = 0; e < NMAX; ++e) acc[j][e] = 0.0f;
        const int t0 = tb + tg * TOKW;
        float rs[TOKW];
#pragma unroll
        for (int j = 0; j < TOKW; ++j) rs[j] = 1.0f;
        if constexpr (NORM) {
            // sum of squares of this warp's quarter of each row, then over lanes
            // (butterfly) and quarters (in q order)
            float ss[TOKW];
#pragma unroll
            for (int j = 0; j < TOKW; ++j) ss[j] = 0.0f;
            for (int sg = q; sg * 256 < d; sg += FR_DS) {
                const int j0 = sg * 256 + 4 * lane;
#pragma unroll
                for (int j = 0; j < TOKW; ++j) {
                    const TX* row = x + static_cast<size_t>(t0 + j) * d;
                    const bool tv = t0 + j < t_end;
                    Raw4<TX> r0, r1;
                    load_raw4(row, j0, tv && j0 < d, r0);
                    load_raw4(row, j0 + 128, tv && j0 + 128 < d, r1);
                    float u[8];
                    unpack_raw4(r0, &u[0]);
                    unpack_raw4(r1, &u[4]);
#pragma unroll
                    for (int k = 0; k < 8; ++k) ss[j] = fmaf(u[k], u[k], ss[j]);
                }
            }
#pragma unroll
            for (int j = 0; j < TOKW; ++j) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], off);
                if (lane == 0) s_ss[tg * TOKW + j][q] = ss[j];
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < TOKW; ++j) {
                float tot = 0.0f;
#pragma unroll
                for (int qq = 0; qq < FR_DS; ++qq) tot += s_ss[tg * TOKW + j][qq];
                rs[j] = 1.0f / sqrtf(tot / static_cast<float>(d) + p.norm_eps);
                if (q == 0 && lane == 0 && t0 + j < t_end) p.rstd[t0 + j] = rs[j];
            }
            if (SMALL) rs_small = rs[0];
        }
        // x of the first segment; inside the loop the next segment's loads are
        // issued before the current one is used
        Raw4<TX> rx[TOKW][2];
#pragma unroll
        for (int j = 0; j < TOKW; ++j) {
            const TX* row = x + static_cast<size_t>(t0 + j) * d;
            const bool tv = t0 + j < t_end;
            const int j0 = q * 256 + 4 * lane;
            load_raw4(row, j0, tv && j0 < d, rx[j][0]);
            load_raw4(row, j0 + 128, tv && j0 + 128 < d, rx[j][1]);
        }
        for (int sg = q; sg * 256 < d; sg += FR_DS) {
            const int j0 = sg * 256 + 4 * lane, j1 = j0 + 128;
            const bool h0 = j0 < d, h1 = j1 < d;
            float xv[TOKW][8];
#pragma unroll
            for (int j = 0; j < TOKW; ++j) {
                unpack_raw4(rx[j][0], &xv[j][0]);
                unpack_raw4(rx[j][1], &xv[j][4]);
                if constexpr (NORM) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) xv[j][k] = scale_round<TX>(xv[j][k], rs[j]);
                }
            }
            const int jn = j0 + FR_DS * 256;
#pragma unroll
            for (int j = 0; j < TOKW; ++j) {
                const TX* row = x + static_cast<size_t>(t0 + j) * d;
                const bool tv = t0 + j < t_end;
                load_raw4(row, jn, tv && jn < d, rx[j][0]);
                load_raw4(row, jn + 128, tv && jn + 128 < d, rx[j][1]);
            }
#pragma unroll
            for (int e = 0; e < NMAX; ++e) {
                if (e < n) {
                    const float* w = wg_s + static_cast<size_t>(e) * d;
                    float4 w0 = make_float4(0.f, 0.f, 0.f, 0.f), w1 = w0;
                    if (SMALL) {
                        if (WPRE && sg == q) {
                            w0 = wpre[WPRE ? e : 0][0];
                            w1 = wpre[WPRE ? e : 0][1];
                        } else {
                            if (h0) w0 = __ldg(reinterpret_cast<const float4*>(w + j0));
                            if (h1) w1 = __ldg(reinterpret_cast<const float4*>(w + j1));
                        }
                    } else {
                        if (h0) w0 = *reinterpret_cast<const float4*>(w + j0);
                        if (h1) w1 = *reinterpret_cast<const float4*>(w + j1);
                    }
                    const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                    for (int j = 0; j < TOKW; ++j) {
                        float a = acc[j][e];
#pragma unroll
                        for (int u = 0; u < 8; ++u) a = fmaf(xv[j][u], wv[u], a);
                        acc[j][e] = a;
                    }
                }
            }
        }
        float v[V];
#pragma unroll
        for (int j = 0; j < TOKW; ++j)
#pragma unroll
            for (int e = 0; e < NMAX; ++e) v[j * NMAX + e] = acc[j][e];
        lane_transpose_sum<V>(v, lane);
        constexpr int VF = V >= 32 ? V / 32 : 1;
#pragma unroll
        for (int i = 0; i < VF; ++i) {
            const int idx = fr_index<V>(lane, i);   // = j * NMAX + e of this warp's tokens
            red[(q * TPB + tg * TOKW) * NMAX + idx] = v[i];
        }
        __syncthreads();
        for (int j = warp; j < TPB; j += FR_WARPS) {
            const int t = tb + j;
            if (t < t_end) {
                float l[NMAX];
#pragma unroll
                for (int e = 0; e < NMAX; ++e) {
                    float s = 0.0f;
                    if (e < n) {
#pragma unroll
                        for (int qq = 0; qq < FR_DS; ++qq) s += red[(qq * TPB + j) * NMAX + e];
                        if (p.bias) s += __ldg(p.bias + e);
                    }
                    l[e] = s;
                }
                topk_gate_write<NMAX>(l, n, K, t, lane, p.topk_idx, p.topk_w, p.logits, s_hist,
                                      SMALL ? s_topk : nullptr);
            }
        }
        __syncthreads();
    }

    // ---------------- grid barrier: publish and collect the block counts ----------------
    // (one block: nothing to exchange; its own counts are the totals)
    int* cnt_word = p.xchg;
    int* gen_word = p.xchg + 1;
    int* bcounts = p.xchg + 2;
    if (G > 1 && tid < 32) bcounts[b * 32 + tid] = tid < n ? s_hist[tid] : 0;
    __syncthreads();
    if (G == 1) {
        if (tid == 0) s_ok = 1;
    } else if (tid == 0) {
        const int g = ld_acquire_gpu(gen_word);
        __threadfence();
        const int prev = atomicAdd(cnt_word, 1);
        int ok = 1;
        if (prev == G - 1) {
            atomicExch(cnt_word, 0);
            __threadfence();
            st_release_gpu(gen_word, g + 1);
        } else {
            const uint64_t t0 = globaltimer_ns();
            uint32_t it = 0;
            while (ld_acquire_gpu(gen_word) == g) {
                if ((++it & 63u) == 0 && globaltimer_ns() - t0 > p.st.wait_ns) {
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    if (!s_ok) {
        if (tid == 0) report(p.st, kStatusTimeout);
        return;
    }
    // Every block has passed the barrier: later kernels may start their prologues.
    griddep_launch_dependents();

    // ---------------- phase 2: offsets, stable positions, row gather ----------------
    // Totals and this block's prefix per expert: warp w sums expert w (and
    // w + 16) over the blocks, lane-strided, then across lanes (integer sums:
    // the order does not matter).
    for (int e = warp; e < n; e += FR_WARPS) {
        int tot = 0, pre = 0;
        if (G == 1) {
            tot = lane == 0 ? s_hist[e] : 0;
        } else {
            for (int bb = lane; bb < G; bb += 32) {
                const int c = __ldcg(bcounts + bb * 32 + e);
                tot += c;
                pre += bb < b ? c : 0;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            tot += __shfl_xor_sync(0xffffffffu, tot, off);
            pre += __shfl_xor_sync(0xffffffffu, pre, off);
        }
        if (lane == 0) {
            s_cnt[e] = tot;
            s_pre[e] = pre;
        }
    }
    if (tid < 32) s_run[tid] = 0;
    __syncthreads();
    if (tid == 0) {
        int running = 0, tp = 0;
        for (int e = 0; e < n; ++e) {
            const int c = s_cnt[e];
            s_base[e] = running + s_pre[e];
            if (b == 0) {
                p.sched[e] = c;
                p.sched[n + e] = running;
                p.sched[2 * n + 1 + e] = tp;
            }
            running += c;
            tp += (c + kTileM - 1) / kTileM;
        }
        if (b == 0) {
            p.sched[2 * n] = running;
            p.sched[3 * n + 1] = tp;
        }
    }
    __syncthreads();

    int2* placed = reinterpret_cast<int2*>(fr_smem);   // [FR_ROUND]; W_g is no longer read
    const int a_begin = t_begin * K, a_end = t_end * K;
    const unsigned lt_mask = (1u << lane) - 1u;
    const uint4* xv4 = static_cast<const uint4*>(p.x);
    uint4* xp4 = static_cast<uint4*>(p.Xp);
    const int R = p.T * K;
    for (int a0 = a_begin; a0 < a_end; a0 += FR_ROUND) {
        const int a = a0 + tid;
        int e = a < a_end ? (SMALL ? s_topk[a - a_begin] : p.topk_idx[a]) : -1;   // this block's phase-1 choices
        // Index checks on every placement (one compare each): an expert id
        // outside [0, n) or a position outside [0, K*T) is never used as an
        // address; the call records MOE_ERR_BOUNDS in the status word instead.
        bool bad = a < a_end && (e < 0 || e >= n);
        if (bad) e = -1;
        wtab[warp][lane] = 0;
        __syncwarp();
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(same & lt_mask);
        if (e >= 0 && rank == 0) wtab[warp][e] = __popc(same);
        __syncthreads();
        // per expert: exclusive scan of the 16 warps' counts, in warp order
        for (int ee = warp; ee < n; ee += FR_WARPS) {
            const int cnt = lane < FR_WARPS ? wtab[lane][ee] : 0;
            const int run = s_run[ee];
            int incl = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += o;
            }
            if (lane < FR_WARPS) wtab[lane][ee] = run + incl - cnt;
            __syncwarp();
            if (lane == 31) s_run[ee] = run + incl;
        }
        __syncthreads();
        if (e >= 0) {
            const int pos = s_base[e] + wtab[warp][e] + rank;
            if (pos >= 0 && pos < R) {
                p.perm[pos] = a;
                p.inv[a] = pos;
                placed[tid] = make_int2(a, pos);
            } else {
                bad = true;
            }
        }
        if (bad) {
            placed[tid] = make_int2(a, -1);
            report(p.st, kStatusBounds);
        }
        __syncthreads();
        if (xp4) {
            const int nr = min(FR_ROUND, a_end - a0);
            const int rv = p.row_vecs;
            // one row per warp at a time, up to 16 x 16 bytes in flight per lane
            // (a whole 8 KB bf16 row of the Mixtral shape)
            for (int r = warp; r < nr; r += FR_WARPS) {
                const int2 ap = placed[r];
                if (ap.y < 0) continue;
                const int t = ap.x / K;
                const uint4* src = xv4 + static_cast<size_t>(t) * rv;
                uint4* dst = xp4 + static_cast<size_t>(ap.y) * rv;
                float rsv = 1.0f;
                if constexpr (NORM) rsv = SMALL ? rs_small : p.rstd[t];   // this block's phase-1 value
                for (int v0 = lane; v0 < rv; v0 += 32 * 16) {
                    uint4 buf[16];
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int vv = v0 + 32 * u;
                        if (vv < rv) buf[u] = __ldg(src + vv);
                    }
                    if constexpr (NORM) {
#pragma unroll
                        for (int u = 0; u < 16; ++u) buf[u] = scale_row_vec<TX>(buf[u], rsv);
                    }
#pragma unroll
                    for (int u = 0; u < 16; ++u) {
                        const int vv = v0 + 32 * u;
                        if (vv < rv) dst[vv] = buf[u];
                    }
                }
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// host side

int fused_route_blocks(int T, int num_sms) {
    if (T <= 0) return 0;
    int g = num_sms < kFusedRouteMaxBlocks ? num_sms : kFusedRouteMaxBlocks;
    if (g > T) g = T;
    const int chunk = (T + g - 1) / g;
    return (T + chunk - 1) / chunk;
}

template <typename TX, int NMAX, int TOKW, bool NORM, bool SMALL>
static cudaError_t launch_fused_s(FusedRouteArgs& a, int G, cudaStream_t s) {
    constexpr int DS = SMALL ? FR_WARPS : FR_DS_LARGE;
    constexpr int TPB = (FR_WARPS / DS) * TOKW;
    const size_t wg_bytes = SMALL ? 0 : static_cast<size_t>(a.n) * a.d * 4;
    const size_t p2_bytes = FR_ROUND * sizeof(int2);
    size_t base = wg_bytes > p2_bytes ? wg_bytes : p2_bytes;
    base = (base + 15) & ~static_cast<size_t>(15);
    a.red_off = base;
    const size_t smem = base + static_cast<size_t>(DS) * TPB * NMAX * 4;
    auto kern = route_fused_kernel<TX, NMAX, TOKW, NORM, SMALL>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(G), dim3(FR_THREADS), smem, s, a);
}

template <typename TX, int NMAX, int TOKW, bool NORM>
static cudaError_t launch_fused_n(FusedRouteArgs& a, int G, cudaStream_t s) {
    if (a.chunk == 1) return launch_fused_s<TX, NMAX, 1, NORM, true>(a, G, s);
    return launch_fused_s<TX, NMAX, TOKW, NORM, false>(a, G, s);
}

template <typename TX, int NMAX, int TOKW>
static cudaError_t launch_fused_t(FusedRouteArgs& a, int G, cudaStream_t s) {
    if (a.rstd) return launch_fused_n<TX, NMAX, TOKW, true>(a, G, s);
    return launch_fused_n<TX, NMAX, TOKW, false>(a, G, s);
}

cudaError_t launch_fused_route(ElemType et, const void* x, const float* Wg, const float* bias, int T, int d, int n,
                               int K, int32_t* topk_idx, float* topk_w, float* logits, int* sched, int32_t* perm,
                               int32_t* inv, void* Xp, int* xchg, float norm_eps, float* rstd, KStatus st,
                               int num_sms, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    if (n > 32) return cudaErrorInvalidValue;
    const int G = fused_route_blocks(T, num_sms);
    FusedRouteArgs a{};
    a.x = x;
    a.Wg = Wg;
    a.bias = bias;
    a.T = T;
    a.d = d;
    a.n = n;
    a.K = K;
    a.chunk = (T + G - 1) / G;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.logits = logits;
    a.sched = sched;
    a.perm = perm;
    a.inv = inv;
    a.Xp = Xp;
    a.row_vecs = d * (et == ElemType::BF16 ? 2 : 4) / 16;
    a.xchg = xchg;
    a.norm_eps = norm_eps;
    a.rstd = rstd;
    a.st = st;
    if (et == ElemType::BF16) {
        if (n <= 8) return launch_fused_t<__nv_bfloat16, 8, 4>(a, G, s);
        if (n <= 16) return launch_fused_t<__nv_bfloat16, 16, 2>(a, G, s);
        return launch_fused_t<__nv_bfloat16, 32, 1>(a, G, s);
    }
    if (n <= 8) return launch_fused_t<float, 8, 4>(a, G, s);
    if (n <= 16) return launch_fused_t<float, 16, 2>(a, G, s);
    return launch_fused_t<float, 32, 1>(a, G, s);
}

}  // namespace moe
