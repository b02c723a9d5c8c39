// decode_fp8.cu -- the weight-streaming expert GEMMs of decode_tc.cu with fp8
// (e4m3) expert weights: one byte per weight read from HBM instead of two,
// for the small batches whose layer time is the time to stream the touched
// experts' weights.
//
// A weight is w = s * q, q an e4m3 value and s one fp32 scale per weight row
// (output feature).  Every e4m3 value is exactly a bf16 value, so each loaded
// tile is widened to bf16 in shared memory and fed to the same bf16 tcgen05
// MMAs as decode_tc.cu (weights as M, the expert's tokens as N, K split S
// ways, identical split choice and K order); the row scale multiplies the fp32
// accumulator row in the epilogue.  When every s is a power of two that product
// is exact and scaling all of one row's products by s commutes with the
// accumulation, so the partial sums -- and everything after them -- equal, bit
// for bit, those of decode_tc.cu run on the bf16 weights s * q.
//
// Widening one byte b = [sign | eeee | mmm]: placing sign at bf16 bit 15 and
// eeeemmm at bits 4..10 gives the bf16 number whose exponent field is eeee,
// i.e. the e4m3 value times 2^-120 (e4m3 bias 7, bf16 bias 127; e4m3
// subnormals, eeee = 0, land on bf16 subnormals with the same mantissa).  One
// bf16 multiply by 2^120 restores the value exactly.  The two NaN bytes (0x7F,
// 0xFF) are outside the accepted input and widen to +-480.
//
// Roles (14 warps):
//   warp 0, lane 0   TMA: the fp8 weight tiles (128 rows x 64 bytes, no
//                    swizzle) and the k-step's token rows (bf16, 128-byte
//                    swizzle) into one stage of a deep ring;
//   warps 6-13       widen a stage's weight tiles into a two-stage bf16 ring in
//                    the 128-byte-swizzled K-major layout the MMA reads;
//   warp 1           owns tensor memory; lane 0 issues the MMAs (A from the
//                    bf16 ring, B = the tokens still in the fp8 stage);
//   warps 2-5        scale and copy finished accumulators to the fp32 partial
//                    sums (two accumulator sets in flight).
// A fp8 stage is free once the converters have read its weights and the MMAs
// that read its tokens have completed.  Every wait is bounded.
#include "kernels.h"

namespace moe {

namespace {
constexpr int Q8_BK = 64;                     // K per stage
constexpr int Q8_UMMA_K = 16;
constexpr int Q8_F8_BYTES = 128 * Q8_BK;      // one fp8 weight tile, 8 KB
constexpr int Q8_BF_BYTES = 128 * Q8_BK * 2;  // the same tile widened, 16 KB
constexpr int Q8_B_BOX = 32;                  // token rows per TMA box
constexpr int Q8_CONV_WARP0 = 6;
constexpr int Q8_CONV_WARPS = 8;
constexpr int Q8_CONV_THREADS = Q8_CONV_WARPS * 32;
constexpr int Q8_THREADS = (Q8_CONV_WARP0 + Q8_CONV_WARPS) * 32;
constexpr int Q8_EPI_THREADS = 128;
constexpr int Q8_MAX_EXPERTS = 32;
constexpr int Q8_MAX_STAGES = 12;
constexpr int Q8_BF_STAGES = 2;
constexpr int Q8_NUM_BARS = 2 * Q8_MAX_STAGES + 2 * Q8_BF_STAGES + 2 + 2 + 1;
constexpr int Q8_TMEM_COLS = 512;
constexpr size_t Q8_SMEM_LIMIT = 227 * 1024;
}  // namespace

struct Fp8DecArgs {
    const int* sched;
    int n;
    int row_blocks;       // weight rows per expert / 128
    int rows_per_e;       // weight rows per expert (F for MODE 0, d for MODE 1)
    int splits;           // S
    int kb_per_split;     // K / 64 / S
    int n_max;            // largest token count per item, rounded up to 32 (<= 256)
    int stages;           // fp8 ring depth
    int stage_bytes;      // fp8 weight tiles + token rows
    int acc_stride;       // TMEM columns per accumulator set
    int acc_sets;         // 1 or 2
    const float* scale0;  // row scales of W1 (MODE 0) or W2 (MODE 1), [n][rows_per_e]
    const float* scale1;  // row scales of W3 (MODE 0)
    float* Pa;            // [S][R][ld] partial sums (MODE 1: the only output)
    float* Pb;            // [S][R][ld] (MODE 0 only)
    int R;
    int ld;               // output features (F for MODE 0, d for MODE 1)
    KStatus st;
};

static size_t fp8_smem_bytes(int a_tiles, int stages, int stage_bytes) {
    return 1024 + static_cast<size_t>(stages) * stage_bytes +
           static_cast<size_t>(Q8_BF_STAGES) * a_tiles * Q8_BF_BYTES + Q8_NUM_BARS * 8 + 16 +
           (3 * Q8_MAX_EXPERTS + 2) * 4 + Q8_MAX_EXPERTS * 4;
}

// bf16x2 product, round to nearest (exact for the widened e4m3 values).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Four e4m3 bytes (element order: low byte first) -> four bf16 in two words.
__device__ __forceinline__ void widen_e4m3x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    constexpr uint32_t kTwo120 = 0x7B807B80u;   // bf16 2^120 in both halves
    const uint32_t mag = w & 0x7F7F7F7Fu, sgn = w & 0x80808080u;
    // magnitudes to bytes 0 and 2 (shifted up by 4 below), signs to bytes 1 and 3
    const uint32_t m01 = __byte_perm(mag, 0u, 0x4140), s01 = __byte_perm(sgn, 0u, 0x1404);
    const uint32_t m23 = __byte_perm(mag, 0u, 0x4342), s23 = __byte_perm(sgn, 0u, 0x3424);
    lo = mul_bf16x2(m01 * 16u + s01, kTwo120);
    hi = mul_bf16x2(m23 * 16u + s23, kTwo120);
}

template <int MODE>
__global__ void __launch_bounds__(Q8_THREADS, 1)
    tc_decode_fp8_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                         const __grid_constant__ CUtensorMap tmB, Fp8DecArgs p) {
    constexpr int A_TILES = MODE == 0 ? 2 : 1;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base_u32 - raw_u32);
    const int FS = p.stages;
    // [FS][stage: A_TILES fp8 tiles, then n_max token rows] [2][A_TILES bf16 tiles]
    const uint32_t ring_u32 = base_u32;
    const uint32_t bf_u32 = ring_u32 + static_cast<uint32_t>(FS * p.stage_bytes);
    const uint8_t* ring_ptr = base_ptr;
    uint8_t* bf_ptr = base_ptr + FS * p.stage_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(bf_ptr + Q8_BF_STAGES * A_TILES * Q8_BF_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Q8_NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_sched = reinterpret_cast<int*>(tmem_slot + 4);
    int* s_touched = s_sched + 3 * Q8_MAX_EXPERTS + 2;

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (Q8_MAX_STAGES + s); };
    auto bfull_bar = [&](int s) { return bar0 + 8u * (2 * Q8_MAX_STAGES + s); };
    auto bempty_bar = [&](int s) { return bar0 + 8u * (2 * Q8_MAX_STAGES + Q8_BF_STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * Q8_MAX_STAGES + 2 * Q8_BF_STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * Q8_MAX_STAGES + 2 * Q8_BF_STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * Q8_MAX_STAGES + 2 * Q8_BF_STAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = p.n;
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < FS; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), Q8_CONV_WARPS + 1);   // converter warps + the MMA commit
        }
        for (int s = 0; s < Q8_BF_STAGES; ++s) {
            mbar_init(bfull_bar(s), Q8_CONV_WARPS);
            mbar_init(bempty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), Q8_EPI_THREADS);
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
        tmem_alloc(smem_u32(tmem_slot), Q8_TMEM_COLS);
        tmem_relinquish();
    }
    // Nothing above reads a buffer of the layer; the schedule and the token
    // rows come from the kernels before this one.
    griddep_wait();
    for (int i = threadIdx.x; i < 3 * n + 2; i += Q8_THREADS) s_sched[i] = p.sched[i];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        int nt = 0;
        for (int e = 0; e < n; ++e)
            if (s_sched[e] > 0) s_touched[nt++] = e;
        s_touched[Q8_MAX_EXPERTS - 1] = nt;   // count kept in the last slot (n <= 31)
    }
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int* counts = s_sched;
    const int* offsets = s_sched + n;
    const int n_touched = s_touched[Q8_MAX_EXPERTS - 1];
    const int items = n_touched * p.row_blocks * p.splits;
    const KStatus st = p.st;

    // item -> (expert, weight row block, K split); K split varies fastest
    auto decode_item = [&](int it, int& e, int& rb, int& sp) {
        sp = it % p.splits;
        const int r = it / p.splits;
        rb = r % p.row_blocks;
        e = s_touched[r / p.row_blocks];
    };
    auto item_n = [&](int e) {
        const int c = counts[e];
        const int nn = (c + Q8_B_BOX - 1) / Q8_B_BOX * Q8_B_BOX;
        return nn < Q8_B_BOX ? Q8_B_BOX : nn;
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
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                int e, rb, sp;
                decode_item(it, e, rb, sp);
                const int nbox = item_n(e) / Q8_B_BOX;
                const int arow = e * p.rows_per_e + rb * 128;
                const int brow = offsets[e];
                const uint32_t bytes = A_TILES * Q8_F8_BYTES + nbox * Q8_B_BOX * Q8_BK * 2;
                for (int kb = sp * p.kb_per_split; kb < (sp + 1) * p.kb_per_split; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, st, abort_flag)) { ok = false; break; }
                    const uint32_t a_dst = ring_u32 + stage * p.stage_bytes;
                    const uint32_t b_dst = a_dst + A_TILES * Q8_F8_BYTES;
                    mbar_arrive_expect_tx(full_bar(stage), bytes);
                    tma_load_2d(a_dst, &tmA0, full_bar(stage), kb * Q8_BK, arow, pol_w);
                    if (MODE == 0) tma_load_2d(a_dst + Q8_F8_BYTES, &tmA1, full_bar(stage), kb * Q8_BK, arow, pol_w);
                    for (int bb = 0; bb < nbox; ++bb)
                        tma_load_2d(b_dst + bb * Q8_B_BOX * Q8_BK * 2, &tmB, full_bar(stage), kb * Q8_BK,
                                    brow + bb * Q8_B_BOX, pol_x);
                    ++issued;
                    if (++stage == FS) { stage = 0; phase ^= 1u; }
                }
            }
            if (!ok) {
                report(st, kStatusTimeout);
                *abort_flag = 1;
            }
            if (*abort_flag) {
                // every stage's most recent load must land before the CTA exits
                for (int s = 0; s < FS; ++s) {
                    if (issued <= s) continue;
                    const long long last = issued - 1 - ((issued - 1 - s) % FS);
                    mbar_wait(full_bar(s), static_cast<uint32_t>((last / FS) & 1), st, nullptr);
                }
            }
        }
        __syncwarp();
    } else if (warp >= Q8_CONV_WARP0) {
        // ---------------- converters: fp8 tiles -> bf16 tiles (128-byte swizzle) ----------------
        // Thread ct widens 16-byte chunks ct and ct + 256 of each 8 KB tile: a
        // warp reads 512 contiguous bytes and writes eight whole bf16 rows, both
        // free of bank conflicts.
        const int ct = threadIdx.x - Q8_CONV_WARP0 * 32;
        int stage = 0, bst = 0;
        uint32_t phase = 0, bph = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
            for (int k = 0; k < p.kb_per_split; ++k) {
                if (!mbar_wait(full_bar(stage), phase, st, abort_flag)) { ok = false; break; }
                if (!mbar_wait(bempty_bar(bst), bph ^ 1u, st, abort_flag)) { ok = false; break; }
                const uint8_t* src = ring_ptr + stage * p.stage_bytes;
                uint8_t* dst = bf_ptr + bst * (A_TILES * Q8_BF_BYTES);
#pragma unroll
                for (int t = 0; t < A_TILES; ++t) {
                    uint4 v[2];
#pragma unroll
                    for (int i = 0; i < 2; ++i)
                        v[i] = *reinterpret_cast<const uint4*>(src + t * Q8_F8_BYTES + (ct + Q8_CONV_THREADS * i) * 16);
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        // chunk c: row c / 4, K elements 16 * (c % 4) .. + 16
                        const int c = ct + Q8_CONV_THREADS * i;
                        const int r = c >> 2, cc = c & 3;
                        uint32_t o[8];
                        widen_e4m3x4(v[i].x, o[0], o[1]);
                        widen_e4m3x4(v[i].y, o[2], o[3]);
                        widen_e4m3x4(v[i].z, o[4], o[5]);
                        widen_e4m3x4(v[i].w, o[6], o[7]);
                        // a bf16 row is 128 bytes = 8 chunks of 16; chunk j sits at j ^ (r % 8)
                        uint8_t* row = dst + t * Q8_BF_BYTES + r * 128;
                        *reinterpret_cast<uint4*>(row + (((2 * cc) ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<uint4*>(row + (((2 * cc + 1) ^ (r & 7)) << 4)) =
                            make_uint4(o[4], o[5], o[6], o[7]);
                    }
                }
                fence_async_shared();   // these generic-proxy writes, before the tensor core reads them
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(empty_bar(stage));
                    mbar_arrive(bfull_bar(bst));
                }
                if (++stage == FS) { stage = 0; phase ^= 1u; }
                if (++bst == Q8_BF_STAGES) { bst = 0; bph ^= 1u; }
            }
        }
        if (!ok) {
            if (lane == 0) report(st, kStatusTimeout);
            *abort_flag = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0, bst = 0;
            uint32_t phase = 0, bph = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                int e, rb, sp;
                decode_item(it, e, rb, sp);
                const int N = item_n(e);
                const uint32_t idesc = idesc_bf16_f32(128, N);
                if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, st, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * p.acc_stride);
                const uint32_t d1 = d0 + static_cast<uint32_t>(p.n_max);
                for (int k = 0; k < p.kb_per_split; ++k) {
                    if (!mbar_wait(bfull_bar(bst), bph, st, abort_flag)) { ok = false; break; }
                    // the token rows' TMA completed on this stage's full barrier
                    if (!mbar_wait(full_bar(stage), phase, st, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = bf_u32 + static_cast<uint32_t>(bst * A_TILES * Q8_BF_BYTES);
                    const uint64_t adesc0 = sdesc_kmajor_sw128(a_addr);
                    const uint64_t adesc1 = sdesc_kmajor_sw128(a_addr + Q8_BF_BYTES);
                    const uint64_t bdesc =
                        sdesc_kmajor_sw128(ring_u32 + static_cast<uint32_t>(stage * p.stage_bytes + A_TILES * Q8_F8_BYTES));
#pragma unroll
                    for (int kk = 0; kk < Q8_BK / Q8_UMMA_K; ++kk) {
                        const uint32_t accum = (k | kk) != 0;
                        mma_bf16_ss(d0, adesc0 + 2u * kk, bdesc + 2u * kk, idesc, accum);
                        if (MODE == 0) mma_bf16_ss(d1, adesc1 + 2u * kk, bdesc + 2u * kk, idesc, accum);
                    }
                    mma_commit(bempty_bar(bst));
                    mma_commit(empty_bar(stage));
                    if (++stage == FS) { stage = 0; phase ^= 1u; }
                    if (++bst == Q8_BF_STAGES) { bst = 0; bph ^= 1u; }
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
        // ---------------- epilogue (warps 2-5): row scale x accumulator -> fp32 partial sums ----------------
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < items; it += gridDim.x) {
            int e, rb, sp;
            decode_item(it, e, rb, sp);
            const int N = item_n(e);
            const int cnt = counts[e];
            const int off = offsets[e];
            const int feat = rb * 128 + q * 32 + lane;   // this thread's weight row = output feature
            const size_t srow = static_cast<size_t>(e) * p.rows_per_e + feat;
            const float sc0 = __ldg(p.scale0 + srow);
            const float sc1 = MODE == 0 ? __ldg(p.scale1 + srow) : 0.0f;
            if (!mbar_wait(accf_bar(acc), acc_phase, st, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
            const uint32_t t0 = tmem_base + static_cast<uint32_t>(acc * p.acc_stride) + lane_off;
#pragma unroll
            for (int part = 0; part < A_TILES; ++part) {
                const float sc = part == 0 ? sc0 : sc1;
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
                        if (j < jn) dst[static_cast<size_t>(j) * p.ld] = sc * __uint_as_float(v[j]);
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
        tmem_dealloc(tmem_base, Q8_TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side

static bool fp8_layout(int mode, int n_max, int& stages, int& stage_bytes, int& acc_stride, int& acc_sets) {
    const int a_tiles = mode == 0 ? 2 : 1;
    stage_bytes = a_tiles * Q8_F8_BYTES + n_max * Q8_BK * 2;   // a multiple of 4 KB
    const size_t fixed = fp8_smem_bytes(a_tiles, 0, stage_bytes);
    stages = static_cast<int>((Q8_SMEM_LIMIT - fixed) / stage_bytes);
    if (stages > Q8_MAX_STAGES) stages = Q8_MAX_STAGES;
    if (stages < 2) return false;
    acc_stride = a_tiles * n_max;
    acc_sets = (2 * acc_stride <= Q8_TMEM_COLS) ? 2 : 1;
    return acc_stride <= Q8_TMEM_COLS;
}

template <int MODE>
static cudaError_t launch_fp8(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b, Fp8DecArgs args,
                              int num_sms, cudaStream_t s) {
    if (!fp8_layout(MODE, args.n_max, args.stages, args.stage_bytes, args.acc_stride, args.acc_sets))
        return cudaErrorInvalidValue;
    const size_t smem = fp8_smem_bytes(MODE == 0 ? 2 : 1, args.stages, args.stage_bytes);
    auto kern = tc_decode_fp8_kernel<MODE>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(num_sms), dim3(Q8_THREADS), smem, s, a0, a1, b, args);
}

cudaError_t launch_decode_fp8_w13(const CUtensorMap& mapW1q, const CUtensorMap& mapW3q, const CUtensorMap& mapXp32,
                                  const float* W1s, const float* W3s, const int* sched, int n, int d, int F, int T,
                                  int K, int splits, float* Pa, float* Pb, KStatus st, int num_sms, cudaStream_t s) {
    if (n > Q8_MAX_EXPERTS - 1 || T <= 0 || T > kDecodeMaxT) return cudaErrorInvalidValue;
    Fp8DecArgs args{};
    args.sched = sched;
    args.n = n;
    args.row_blocks = F / 128;
    args.rows_per_e = F;
    args.splits = splits;
    args.kb_per_split = d / Q8_BK / splits;
    args.n_max = (T + Q8_B_BOX - 1) / Q8_B_BOX * Q8_B_BOX;
    args.scale0 = W1s;
    args.scale1 = W3s;
    args.Pa = Pa;
    args.Pb = Pb;
    args.R = K * T;
    args.ld = F;
    args.st = st;
    return launch_fp8<0>(mapW1q, mapW3q, mapXp32, args, num_sms, s);
}

cudaError_t launch_decode_fp8_w2(const CUtensorMap& mapW2q, const CUtensorMap& mapH32, const float* W2s,
                                 const int* sched, int n, int d, int F, int T, int K, int splits, float* P2, KStatus st,
                                 int num_sms, cudaStream_t s) {
    if (n > Q8_MAX_EXPERTS - 1 || T <= 0 || T > kDecodeMaxT) return cudaErrorInvalidValue;
    Fp8DecArgs args{};
    args.sched = sched;
    args.n = n;
    args.row_blocks = d / 128;
    args.rows_per_e = d;
    args.splits = splits;
    args.kb_per_split = F / Q8_BK / splits;
    args.n_max = (T + Q8_B_BOX - 1) / Q8_B_BOX * Q8_B_BOX;
    args.scale0 = W2s;
    args.scale1 = W2s;
    args.Pa = P2;
    args.Pb = nullptr;
    args.R = K * T;
    args.ld = d;
    args.st = st;
    return launch_fp8<1>(mapW2q, mapW2q, mapH32, args, num_sms, s);
}

}  // namespace moe
