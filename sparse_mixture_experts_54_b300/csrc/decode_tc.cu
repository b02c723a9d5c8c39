// decode_tc.cu -- weight-streaming expert GEMMs for small batches.
//
// With few tokens per expert the layer reads every touched expert's weights
// once and does little arithmetic per byte, so it is bound by HBM bandwidth,
// not by the tensor cores (the memory-vs-compute remark of the xyznot
// summary, "Limitations").  These kernels therefore put the weights in the
// MMA's M operand and the expert's tokens in N ("swap-AB"):
//
//   MODE 0:  Da = W1_e[rows] . X_e^T,  Db = W3_e[rows] . X_e^T     (128 weight rows x N tokens)
//   MODE 1:  D  = W2_e[rows] . H_e^T
//
// and split K so that the work spreads evenly over all SMs: by default, from
// two tokens on, every CTA takes an equal, contiguous share of the k-blocks of
// all (touched expert, row block) units laid end to end (stream-K); for one
// token, and when asked, K is cut into S uniform parts per unit (SplitGeom in
// kernels.h).  Each piece writes fp32 partial sums
// P[slot][row of X_e or H_e][output feature]; a small follow-up kernel adds a
// unit's slots in K order (then SiLU(a)*b for MODE 0, or gate, slot sum and
// rounding for MODE 1), so results stay bitwise reproducible.
//
// Pipeline (one CTA per SM, persistent over its pieces): warp 0 lane 0 streams
// weight tiles (128 rows x 64 K, 128-byte swizzle) and token tiles (32 rows x
// 64 K) with TMA into a ring of stages sized to the batch; warp 1 owns tensor
// memory and issues tcgen05.mma (M=128, N = the expert's tokens rounded up to
// 32); warps 2-5 move finished accumulators to the partial buffers, two
// accumulator sets in flight so the copy-out overlaps the next item.  Every
// wait is bounded, as in gemm_tc.cu.
#include "kernels.h"
#include "route_common.cuh"

namespace moe {

namespace {
constexpr int D_BK = 64;
constexpr int D_UMMA_K = 16;
constexpr int D_A_BYTES = 128 * D_BK * 2;   // one 128-row weight tile, 16 KB
constexpr int D_B_BOX = 32;                 // token rows per TMA box
constexpr int D_THREADS = 192;
constexpr int D_EPI_THREADS = 128;
constexpr int D_MAX_EXPERTS = 32;
constexpr int D_MAX_STAGES = 8;
constexpr int D_NUM_BARS = 2 * D_MAX_STAGES + 2 + 2 + 1;
constexpr int D_TMEM_COLS = 512;
}  // namespace

struct DecArgs {
    const int* sched;
    int n;
    int row_blocks;       // weight rows per expert / 128
    int rows_per_e;       // weight rows per expert (F for MODE 0, d for MODE 1)
    int splits;           // S (uniform splits), 0: stream-K (SplitGeom in kernels.h)
    int kb_per_split;     // K / 64 / S (uniform)
    int kb_unit;          // K / 64: k-blocks of a unit
    int n_max;            // largest token count per item, rounded up to 32 (<= 256)
    int stages;
    int stage_bytes;
    int acc_stride;       // TMEM columns per accumulator set
    int acc_sets;         // 1 or 2
    float* Pa;            // [S][R][ld] partial sums (MODE 1: the only output)
    float* Pb;            // [S][R][ld] (MODE 0 only)
    int R;
    int ld;               // output features (F for MODE 0, d for MODE 1)
    // Schedule-ready word (may be null): the routing kernel clears it, MODE 0
    // sets it once it holds the call's schedule, MODE 1 reads it to start its
    // weight loads before the wait on the kernel before it.
    int* ready;
    KStatus st;
};

static size_t decode_smem_bytes(int stages, int stage_bytes) {
    return 1024 + static_cast<size_t>(stages) * stage_bytes + D_NUM_BARS * 8 + 16 + (3 * D_MAX_EXPERTS + 2) * 4 +
           D_MAX_EXPERTS * 4 + 16;
}

template <int MODE>
__global__ void __launch_bounds__(D_THREADS, 1)
    tc_decode_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                     const __grid_constant__ CUtensorMap tmB, DecArgs p) {
    constexpr int A_TILES = MODE == 0 ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t ring_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t* ring_ptr = smem_raw + (ring_u32 - raw_u32);
    uint64_t* bars = reinterpret_cast<uint64_t*>(ring_ptr + static_cast<size_t>(p.stages) * p.stage_bytes);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + D_NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_sched = reinterpret_cast<int*>(tmem_slot + 4);
    int* s_touched = s_sched + 3 * D_MAX_EXPERTS + 2;   // touched experts, in expert order
    int* s_early = s_touched + D_MAX_EXPERTS;           // MODE 1: schedule known before the wait

    const uint32_t bar0 = smem_u32(bars);
    const int S = p.stages;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (D_MAX_STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * D_MAX_STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * D_MAX_STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * D_MAX_STAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = p.n;
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), D_EPI_THREADS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA0);
        if (MODE == 0) tma_prefetch_desc(&tmA1);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), D_TMEM_COLS);
        tmem_relinquish();
    }
    // Everything above touches no buffer of the layer; the schedule and the
    // token rows come from the kernels before this one.
    //
    // W2 (MODE 1) reads H, which the SwiGLU kernel right before it writes, but its
    // weights and schedule are older: the W1/W3 kernel of the same call has set the
    // ready word (release) after its own wait on the routing kernel.  When the word
    // is set, this kernel reads the schedule at once and its producer sends the
    // first ring's worth of weight tiles before waiting for the SwiGLU kernel; only
    // the token rows (H) and everything after wait (the MMA and copy-out roles
    // wait for the SwiGLU kernel as they start).  The routing kernel of every
    // call clears the word once the previous call has finished, so a set word is
    // always this call's.
    bool early = false;
    if (MODE == 1 && p.ready) {
        if (threadIdx.x == 0) {
            // a few microseconds at most; past that the kernel waits as usual
            const uint64_t t0 = globaltimer_ns();
            int v = ld_acquire_gpu(p.ready);
            while (v == 0 && globaltimer_ns() - t0 < 3000) v = ld_acquire_gpu(p.ready);
            *s_early = v;
        }
        __syncthreads();
        early = *s_early != 0;
    }
    if (!early) griddep_wait();
    for (int i = threadIdx.x; i < 3 * n + 2; i += D_THREADS) s_sched[i] = __ldcg(p.sched + i);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (MODE == 0 && p.ready && blockIdx.x == 0 && threadIdx.x == 0) st_release_gpu(p.ready, 1);
    if (threadIdx.x == 0) {
        int nt = 0;
        for (int e = 0; e < n; ++e)
            if (s_sched[e] > 0) s_touched[nt++] = e;
        s_touched[D_MAX_EXPERTS - 1] = nt;   // count kept in the last slot (n <= 31)
    }
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int* counts = s_sched;
    const int* offsets = s_sched + n;
    const int n_touched = s_touched[D_MAX_EXPERTS - 1];
    const KStatus st = p.st;

    // This CTA's work in order: segments (expert, row block, k-blocks [kb0, kb1),
    // partial-sum slot), by the uniform or the stream-K split (SplitGeom).
    const int U = n_touched * p.row_blocks;
    const long long Wk = static_cast<long long>(U) * p.kb_unit;
    const int Gsk = p.splits == 0 ? sk_grid(Wk, p.kb_unit, gridDim.x) : 0;
    struct Seg {
        int e, rb, kb0, kb1, slot;
    };
    auto walk_init = [&](long long& cur, long long& end) {
        if (p.splits == 0) {
            const bool mine = static_cast<int>(blockIdx.x) < Gsk;
            cur = mine ? sk_start(blockIdx.x, Wk, Gsk) : 0;
            end = mine ? sk_start(blockIdx.x + 1, Wk, Gsk) : 0;
        } else {
            cur = blockIdx.x;
            end = static_cast<long long>(U) * p.splits;
        }
    };
    auto walk_next = [&](long long& cur, long long end, Seg& g) -> bool {
        if (cur >= end) return false;
        int u;
        if (p.splits == 0) {
            u = static_cast<int>(cur / p.kb_unit);
            g.kb0 = static_cast<int>(cur % p.kb_unit);
            g.kb1 = static_cast<int>(min(static_cast<long long>(p.kb_unit), g.kb0 + (end - cur)));
            g.slot = static_cast<int>(blockIdx.x) - sk_cta_of(static_cast<long long>(u) * p.kb_unit, Wk, Gsk);
            cur += g.kb1 - g.kb0;
        } else {
            const int it = static_cast<int>(cur);
            u = it / p.splits;
            g.slot = it % p.splits;
            g.kb0 = g.slot * p.kb_per_split;
            g.kb1 = g.kb0 + p.kb_per_split;
            cur += gridDim.x;
        }
        g.rb = u % p.row_blocks;
        g.e = s_touched[u / p.row_blocks];
        return true;
    };
    auto item_n = [&](int e) {
        const int c = counts[e];
        const int nn = (c + D_B_BOX - 1) / D_B_BOX * D_B_BOX;
        return nn < D_B_BOX ? D_B_BOX : nn;
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            const uint64_t pol_w = policy_evict_first();   // each weight byte is read once
            const uint64_t pol_x = policy_evict_last();    // token rows are re-read by every row block
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            // early (MODE 1): the first `pre` stages (first use of the ring, no
            // empty wait) get their byte count and weight tile now; their token
            // rows follow the wait, in the loop below
            int pre = 0;
            long long cur, end;
            Seg g;
            if (early) {
                walk_init(cur, end);
                while (pre < S && walk_next(cur, end, g)) {
                    const int nbox = item_n(g.e) / D_B_BOX;
                    const int arow = g.e * p.rows_per_e + g.rb * 128;
                    const uint32_t bytes = A_TILES * D_A_BYTES + nbox * D_B_BOX * D_BK * 2;
                    for (int kb = g.kb0; kb < g.kb1 && pre < S; ++kb, ++pre) {
                        mbar_arrive_expect_tx(full_bar(pre), bytes);
                        tma_load_2d(ring_u32 + pre * p.stage_bytes, &tmA0, full_bar(pre), kb * D_BK, arow, pol_w);
                    }
                }
                griddep_wait();
            }
            walk_init(cur, end);
            while (ok && walk_next(cur, end, g)) {
                const int nbox = item_n(g.e) / D_B_BOX;
                const int arow = g.e * p.rows_per_e + g.rb * 128;
                const int brow = offsets[g.e];
                const uint32_t bytes = A_TILES * D_A_BYTES + nbox * D_B_BOX * D_BK * 2;
                for (int kb = g.kb0; kb < g.kb1; ++kb) {
                    const uint32_t a_dst = ring_u32 + stage * p.stage_bytes;
                    const uint32_t b_dst = a_dst + A_TILES * D_A_BYTES;
                    if (issued >= pre) {
                        if (!mbar_wait(empty_bar(stage), phase ^ 1u, st, abort_flag)) { ok = false; break; }
                        mbar_arrive_expect_tx(full_bar(stage), bytes);
                        tma_load_2d(a_dst, &tmA0, full_bar(stage), kb * D_BK, arow, pol_w);
                        if (MODE == 0) tma_load_2d(a_dst + D_A_BYTES, &tmA1, full_bar(stage), kb * D_BK, arow, pol_w);
                    }
                    for (int bb = 0; bb < nbox; ++bb)
                        tma_load_2d(b_dst + bb * D_B_BOX * D_BK * 2, &tmB, full_bar(stage), kb * D_BK,
                                    brow + bb * D_B_BOX, pol_x);
                    ++issued;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                report(st, kStatusTimeout);
                *abort_flag = 1;
            }
            if (*abort_flag) {
                // every stage's most recent load must land before the CTA exits
                for (int s = 0; s < S; ++s) {
                    if (issued <= s) continue;
                    const long long last = issued - 1 - ((issued - 1 - s) % S);
                    mbar_wait(full_bar(s), static_cast<uint32_t>((last / S) & 1), st, nullptr);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (early) griddep_wait();   // only the producer's first weight tiles go ahead of it
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            long long cur, end;
            Seg g;
            walk_init(cur, end);
            while (ok && walk_next(cur, end, g)) {
                const int N = item_n(g.e);
                const uint32_t idesc = idesc_bf16_f32(128, N);
                if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, st, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * p.acc_stride);
                const uint32_t d1 = d0 + static_cast<uint32_t>(p.n_max);
                for (int k = 0; k < g.kb1 - g.kb0; ++k) {
                    if (!mbar_wait(full_bar(stage), phase, st, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = ring_u32 + stage * p.stage_bytes;
                    const uint64_t adesc0 = sdesc_kmajor_sw128(a_addr);
                    const uint64_t adesc1 = sdesc_kmajor_sw128(a_addr + D_A_BYTES);
                    const uint64_t bdesc = sdesc_kmajor_sw128(a_addr + A_TILES * D_A_BYTES);
#pragma unroll
                    for (int kk = 0; kk < D_BK / D_UMMA_K; ++kk) {
                        const uint32_t accum = (k | kk) != 0;
                        mma_bf16_ss(d0, adesc0 + 2u * kk, bdesc + 2u * kk, idesc, accum);
                        if (MODE == 0) mma_bf16_ss(d1, adesc1 + 2u * kk, bdesc + 2u * kk, idesc, accum);
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(accf_bar(acc));
                if (++acc == p.acc_sets) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) {
                report(st, kStatusTimeout);
                *abort_flag = 1;
            }
            mma_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, st, nullptr)) report(st, kStatusTimeout);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: accumulator -> fp32 partial sums ----------------
        if (early) griddep_wait();
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        long long cur, end;
        Seg g;
        walk_init(cur, end);
        while (walk_next(cur, end, g)) {
            const int N = item_n(g.e);
            const int cnt = counts[g.e];
            const int off = offsets[g.e];
            const int sp = g.slot;
            if (!mbar_wait_warp(accf_bar(acc), acc_phase, st, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const int feat = g.rb * 128 + q * 32 + lane;   // this thread's weight row = output feature
            const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
            const uint32_t t0 = tmem_base + static_cast<uint32_t>(acc * p.acc_stride) + lane_off;
            for (int part = 0; part < A_TILES; ++part) {
                float* P = (part == 0 ? p.Pa : p.Pb) + static_cast<size_t>(sp) * p.R * p.ld;
                const uint32_t tp = t0 + static_cast<uint32_t>(part * p.n_max);
                for (int c = 0; c < N; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tp + c, v);
                    tmem_ld_wait();
                    const int jn = min(32, cnt - c);
                    float* dst = P + static_cast<size_t>(off + c) * p.ld + feat;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (j < jn) dst[static_cast<size_t>(j) * p.ld] = __uint_as_float(v[j]);
                }
            }
            tc_fence_before();
            mbar_arrive(acce_bar(acc));
            if (++acc == p.acc_sets) {
                acc = 0;
                acc_phase ^= 1u;
            }
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
        tmem_dealloc(tmem_base, D_TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Per-block view of the split geometry (SplitGeom): how many partial-sum slots
// the row block rb of expert e has.  Stream-K needs the call's unit count and
// each expert's rank among the touched ones, from the schedule.
struct SlotMap {
    int sk, S, rbe, n, kb, G;
    long long W;
    int rank[D_MAX_EXPERTS];    // touched rank per expert
    int off[D_MAX_EXPERTS];     // first row per expert
    int cnt[D_MAX_EXPERTS];     // rows per expert
};

// All threads of the block; ends with the block synchronised.
__device__ __forceinline__ void slot_map_init(SlotMap& m, const SplitGeom& g) {
    if (threadIdx.x == 0) {
        m.sk = g.sk;
        m.S = g.S;
        m.rbe = g.rb;
        m.n = g.n;
        m.kb = g.kb;
    }
    if (g.sk && static_cast<int>(threadIdx.x) < g.n) {   // the schedule's words, one per thread
        m.cnt[threadIdx.x] = __ldcg(g.sched + threadIdx.x);
        m.off[threadIdx.x] = __ldcg(g.sched + g.n + threadIdx.x);
    }
    __syncthreads();
    if (!g.sk) return;
    if (threadIdx.x == 0) {
        int nt = 0;
        for (int e = 0; e < g.n; ++e) {
            m.rank[e] = nt;
            nt += m.cnt[e] > 0;
        }
        m.W = static_cast<long long>(nt) * g.rb * g.kb;
        m.G = sk_grid(m.W, g.kb, g.grid);
    }
    __syncthreads();
}

__device__ __forceinline__ int slots_of(const SlotMap& m, int e, int rb) {
    return m.sk ? sk_slots(m.rank[e] * m.rbe + rb, m.W, m.kb, m.G) : m.S;
}

// the expert whose rows hold row r (rows are expert-contiguous)
__device__ __forceinline__ int expert_of_row(const SlotMap& m, int r) {
    int e_sel = 0;
    for (int e = 0; e < m.n; ++e)
        if (m.cnt[e] > 0 && r >= m.off[e]) e_sel = e;
    return e_sel;
}

// H[r][f] = bf16( SiLU(sum_s Pa[s][r][f]) * sum_s Pb[s][r][f] ), parts added in order.
// kBatch: splits per round trip; 2 (at most 2 slots, the larger batches) leaves
// registers for 4 blocks per SM, so a T = 32 layer's 896 blocks fit in one wave.
template <int kBatch>
__global__ void __launch_bounds__(256, kBatch <= 2 ? 4 : 2)
    decode_swiglu_kernel(const float4* __restrict__ Pa, const float4* __restrict__ Pb, SplitGeom geo, int F4,
                         size_t part4, uint2* __restrict__ H) {
    __shared__ SlotMap sm;
    griddep_launch_dependents();
    griddep_wait();
    slot_map_init(sm, geo);
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < part4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        int S = sm.S;
        if (sm.sk) {
            const int r = static_cast<int>(i / F4), rb = static_cast<int>(i % F4) / 32;   // 32 float4 = 128 features
            S = slots_of(sm, expert_of_row(sm, r), rb);
        }
        float4 a, b;
        sum_splits_pair<kBatch>(Pa + i, Pb + i, part4, S, S, a, b);
        uint2 o;
        o.x = pack_bf16x2(silu_f(a.x) * b.x, silu_f(a.y) * b.y);
        o.y = pack_bf16x2(silu_f(a.z) * b.z, silu_f(a.w) * b.w);
        H[i] = o;
    }
}

// y[t][i] = sum_k g[t][k] * (sum_s P2[s][inv[t*K+k]][i]), slots in order, one rounding.
// With resid (may be y itself): y = resid + that sum, one rounding.  PAIR (K = 2,
// small batches): both slot rows' split loads go out together, one round trip
// to L2 per 8 splits instead of two; the registers that takes allow one block
// per SM, which the few blocks of a small batch do not miss.  Same arithmetic
// in the same order either way.  Under stream-K a slot row's split count follows
// its expert (topk_idx) and the row block of the column.
template <typename TY, bool PAIR>
__global__ void __launch_bounds__(256, PAIR ? 1 : 2)
    decode_combine_kernel(const float4* __restrict__ P2, SplitGeom geo, size_t part4, const int32_t* __restrict__ inv,
                          const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w, int T, int K, int d4,
                          const TY* resid, TY* y) {
    __shared__ SlotMap sm;
    griddep_launch_dependents();
    griddep_wait();
    slot_map_init(sm, geo);
    const size_t total = static_cast<size_t>(T) * d4;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t t = i / d4, c = i % d4;
        const int rb = static_cast<int>(c) / 32;   // 32 float4 = 128 output features
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (PAIR) {
            const size_t row0 = static_cast<size_t>(inv[2 * t]), row1 = static_cast<size_t>(inv[2 * t + 1]);
            const float g0 = topk_w[2 * t], g1 = topk_w[2 * t + 1];
            const int S0 = sm.sk ? slots_of(sm, topk_idx[2 * t], rb) : sm.S;
            const int S1 = sm.sk ? slots_of(sm, topk_idx[2 * t + 1], rb) : sm.S;
            float4 v0, v1;
            sum_splits_pair(P2 + row0 * d4 + c, P2 + row1 * d4 + c, part4, S0, S1, v0, v1);
            acc.x = fmaf(g0, v0.x, acc.x); acc.y = fmaf(g0, v0.y, acc.y);
            acc.z = fmaf(g0, v0.z, acc.z); acc.w = fmaf(g0, v0.w, acc.w);
            acc.x = fmaf(g1, v1.x, acc.x); acc.y = fmaf(g1, v1.y, acc.y);
            acc.z = fmaf(g1, v1.z, acc.z); acc.w = fmaf(g1, v1.w, acc.w);
        } else {
            for (int k = 0; k < K; ++k) {
                const size_t a = t * K + k;
                const size_t row = static_cast<size_t>(inv[a]);
                const float g = topk_w[a];
                const int S = sm.sk ? slots_of(sm, topk_idx[a], rb) : sm.S;
                const float4 v = sum_splits(P2 + row * d4 + c, part4, S);
                acc.x = fmaf(g, v.x, acc.x); acc.y = fmaf(g, v.y, acc.y);
                acc.z = fmaf(g, v.z, acc.z); acc.w = fmaf(g, v.w, acc.w);
            }
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
            acc.x = r[0] + acc.x; acc.y = r[1] + acc.y; acc.z = r[2] + acc.z; acc.w = r[3] + acc.w;
        }
        if constexpr (sizeof(TY) == 4) {
            reinterpret_cast<float4*>(y)[i] = acc;
        } else {
            uint2 o;
            o.x = pack_bf16x2(acc.x, acc.y);
            o.y = pack_bf16x2(acc.z, acc.w);
            reinterpret_cast<uint2*>(y)[i] = o;
        }
    }
}

// ---------------------------------------------------------------------------
// host side

// Number of K splits for `units` (expert, row block) pairs: the smallest divisor
// of kblocks (<= kDecodeMaxSplits) whose items fill the SMs' waves to >= 90%,
// else the one that fills them best.  (Fewer, longer items: a 95% threshold
// measured 1-4% slower at T = 8..128 and no faster at T = 1.)
int decode_pick_splits(int units, int kblocks, int num_sms) {
    int best = 1;
    double best_eff = 0.0;
    for (int s = 1; s <= kDecodeMaxSplits; ++s) {
        if (kblocks % s) continue;
        const long long items = static_cast<long long>(units) * s;
        const long long waves = (items + num_sms - 1) / num_sms;
        const double eff = static_cast<double>(items) / static_cast<double>(waves * num_sms);
        if (eff >= 0.90) return s;
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = s;
        }
    }
    return best;
}

static bool decode_layout(int mode, int n_max, int stage_cap, int& stages, int& stage_bytes, int& acc_stride,
                          int& acc_sets) {
    const int a_tiles = mode == 0 ? 2 : 1;
    stage_bytes = a_tiles * D_A_BYTES + n_max * D_BK * 2;
    stages = static_cast<int>((200 * 1024) / stage_bytes);
    if (stages > D_MAX_STAGES) stages = D_MAX_STAGES;
    if (stage_cap > 0 && stages > stage_cap) stages = stage_cap;
    if (stages < 2) return false;
    acc_stride = a_tiles * n_max;
    acc_sets = (2 * acc_stride <= D_TMEM_COLS) ? 2 : 1;
    return acc_stride <= D_TMEM_COLS;
}

template <int MODE>
static cudaError_t launch_decode(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b, DecArgs args,
                                 int num_sms, cudaStream_t s, int stage_cap = 0) {
    if (!decode_layout(MODE, args.n_max, stage_cap, args.stages, args.stage_bytes, args.acc_stride, args.acc_sets))
        return cudaErrorInvalidValue;
    const size_t smem = decode_smem_bytes(args.stages, args.stage_bytes);
    auto kern = tc_decode_kernel<MODE>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(num_sms), dim3(D_THREADS), smem, s, a0, a1, b, args);
}

cudaError_t launch_decode_w13(const CUtensorMap& mapW1, const CUtensorMap& mapW3, const CUtensorMap& mapXp32,
                              const int* sched, int n, int d, int F, int T, int K, int splits, float* Pa, float* Pb,
                              KStatus st, int num_sms, cudaStream_t s, int* ready) {
    if (n > D_MAX_EXPERTS - 1 || T <= 0 || T > kDecodeMaxT) return cudaErrorInvalidValue;
    DecArgs args{};
    args.ready = ready;
    args.sched = sched;
    args.n = n;
    args.row_blocks = F / 128;
    args.rows_per_e = F;
    args.splits = splits;
    args.kb_unit = d / D_BK;
    args.kb_per_split = splits > 0 ? d / D_BK / splits : 0;
    args.n_max = (T + D_B_BOX - 1) / D_B_BOX * D_B_BOX;
    args.Pa = Pa;
    args.Pb = Pb;
    args.R = K * T;
    args.ld = F;
    args.st = st;
    // One token: a 4-stage ring (144 KB) measured 1.4% faster than the 5 that fit
    // 200 KB for a layer call after the L2 is overwritten (133.4 against 135.3 us;
    // the same within 0.2 us in a stack of layers); from 2 tokens on, 5.
    return launch_decode<0>(mapW1, mapW3, mapXp32, args, num_sms, s, T == 1 ? 4 : 0);
}

cudaError_t launch_decode_w2(const CUtensorMap& mapW2, const CUtensorMap& mapH32, const int* sched, int n, int d,
                             int F, int T, int K, int splits, float* P2, KStatus st, int num_sms, cudaStream_t s,
                             int* ready) {
    if (n > D_MAX_EXPERTS - 1 || T <= 0 || T > kDecodeMaxT) return cudaErrorInvalidValue;
    DecArgs args{};
    args.ready = ready;
    args.sched = sched;
    args.n = n;
    args.row_blocks = d / 128;
    args.rows_per_e = d;
    args.splits = splits;
    args.kb_unit = F / D_BK;
    args.kb_per_split = splits > 0 ? F / D_BK / splits : 0;
    args.n_max = (T + D_B_BOX - 1) / D_B_BOX * D_B_BOX;
    args.Pa = P2;
    args.Pb = nullptr;
    args.R = K * T;
    args.ld = d;
    args.st = st;
    return launch_decode<1>(mapW2, mapW2, mapH32, args, num_sms, s);
}

SplitGeom decode_geom(int splits, int kblocks, int row_blocks, const int* sched, int n, int num_sms) {
    SplitGeom g;
    g.sk = splits == 0;
    g.S = splits > 0 ? splits : 1;
    g.kb = kblocks;
    g.rb = row_blocks;
    g.grid = num_sms;
    g.sched = sched;
    g.n = n;
    return g;
}

cudaError_t launch_decode_swiglu(const float* Pa, const float* Pb, const SplitGeom& g, int R, int F,
                                 __nv_bfloat16* H, cudaStream_t s) {
    const size_t part4 = static_cast<size_t>(R) * F / 4;
    int blocks = static_cast<int>((part4 + 255) / 256);
    if (blocks > 148 * 8) blocks = 148 * 8;
    if (blocks < 1) blocks = 1;
    // two splits per round trip: uniform S <= 2, or stream-K (W1/W3 rows split in at
    // most two pieces once the units fill the grid)
    auto kern = (g.sk || g.S <= 2) ? decode_swiglu_kernel<2> : decode_swiglu_kernel<8>;
    return launch_pdl(kern, dim3(blocks), dim3(256), 0, s, reinterpret_cast<const float4*>(Pa),
                      reinterpret_cast<const float4*>(Pb), g, F / 4, part4, reinterpret_cast<uint2*>(H));
}

cudaError_t launch_decode_combine(ElemType et, const float* P2, const SplitGeom& g, int R, const int32_t* inv,
                                  const int32_t* topk_idx, const float* topk_w, int T, int K, int d, const void* resid,
                                  void* y, cudaStream_t s) {
    const size_t part4 = static_cast<size_t>(R) * d / 4;
    const int d4 = d / 4;
    const size_t total = static_cast<size_t>(T) * d4;
    int blocks = static_cast<int>((total + 255) / 256);
    if (blocks > 148 * 8) blocks = 148 * 8;
    if (blocks < 1) blocks = 1;
    // the pair kernel while its threads fit in one wave of one block per SM
    const bool pair = K == 2 && blocks <= 148;
    if (et == ElemType::BF16) {
        auto kern = pair ? decode_combine_kernel<__nv_bfloat16, true> : decode_combine_kernel<__nv_bfloat16, false>;
        return launch_pdl(kern, dim3(blocks), dim3(256), 0, s, reinterpret_cast<const float4*>(P2), g, part4, inv,
                          topk_idx, topk_w, T, K, d4, static_cast<const __nv_bfloat16*>(resid),
                          static_cast<__nv_bfloat16*>(y));
    }
    auto kern = pair ? decode_combine_kernel<float, true> : decode_combine_kernel<float, false>;
    return launch_pdl(kern, dim3(blocks), dim3(256), 0, s, reinterpret_cast<const float4*>(P2), g, part4, inv, topk_idx,
                      topk_w, T, K, d4, static_cast<const float*>(resid), static_cast<float*>(y));
}

}  // namespace moe
