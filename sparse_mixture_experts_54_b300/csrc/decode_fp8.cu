// decode_fp8.cu -- the weight-streaming expert GEMMs of decode_tc.cu with fp8
// (e4m3) expert weights: one byte per weight read from HBM instead of two,
// for the small batches whose layer time is the time to stream the touched
// experts' weights.
//
// A weight is w = s * q, q an e4m3 value and s one fp32 scale per weight row
// (output feature).  Every e4m3 value is exactly a bf16 value, so each loaded
// tile is widened to bf16 on chip and fed to the same bf16 tcgen05 MMAs as
// decode_tc.cu (weights as M = 128 rows, the expert's tokens as N, K split S
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
// The widened weights go to tensor memory, not shared memory: the MMA reads
// its A operand from there, so each weight byte crosses shared memory once
// (TMA write, converter read) instead of four times.
//
// Roles (22 warps):
//   warp 0, lane 0   TMA: the fp8 weight tile(s) of a k-step (128 rows x 64
//                    bytes, 64-byte swizzle) and the k-step's token rows (bf16,
//                    128-byte swizzle) into one stage of a deep shared ring;
//   warps 6-21       widen the weights into a ring of A stages in tensor
//                    memory (tcgen05.st); four warps per lane quadrant, each
//                    thread one weight row;
//   warp 1           owns tensor memory; lane 0 issues the MMAs (A from tensor
//                    memory, B = the tokens in the fp8 stage);
//   warps 2-5        scale and copy finished accumulators to the fp32 partial
//                    sums (two accumulator sets in flight when they fit).
// Tensor memory (512 columns) holds the accumulators, then the A stages; the
// split between them, the shared ring's depth and whether W1 and W3 share an
// item follow the largest per-expert token count, read on the device.  A fp8
// stage is free once the converters have read its weights and the MMAs that
// read its tokens have completed.  Every wait is bounded.
#include "kernels.h"

namespace moe {

namespace {
constexpr int Q8_BK = 64;                     // K per step
constexpr int Q8_UMMA_K = 16;
constexpr int Q8_F8_BYTES = 128 * Q8_BK;      // one fp8 weight tile, 8 KB
constexpr int Q8_B_BOX = 32;                  // token rows per TMA box
constexpr int Q8_CONV_WARP0 = 6;
constexpr int Q8_CONV_WARPS = 16;             // four per tensor-memory lane quadrant
constexpr int Q8_THREADS = (Q8_CONV_WARP0 + Q8_CONV_WARPS) * 32;
constexpr int Q8_EPI_THREADS = 128;
constexpr int Q8_MAX_EXPERTS = 32;
constexpr int Q8_MAX_STAGES = 16;             // fp8 ring in shared memory
constexpr int Q8_MAX_ASTAGES = 8;             // widened-weight ring in tensor memory
constexpr int Q8_NUM_BARS = 2 * Q8_MAX_STAGES + 2 * Q8_MAX_ASTAGES + 2 + 2 + 1;
constexpr int Q8_TMEM_COLS = 512;
constexpr int Q8_TMEM_SPARE = 32;             // columns never used, past the last A stage
constexpr size_t Q8_SMEM_BYTES = 227 * 1024;
constexpr size_t Q8_SMEM_FIXED =
    1024 + Q8_NUM_BARS * 8 + 32 + (3 * Q8_MAX_EXPERTS + 2) * 4 + Q8_MAX_EXPERTS * 4;
constexpr int Q8_RING_BYTES = static_cast<int>((Q8_SMEM_BYTES - Q8_SMEM_FIXED) / 1024 * 1024);
}  // namespace

struct Fp8DecArgs {
    const int* sched;
    int n;
    int row_blocks;       // weight rows per expert / 128
    int rows_per_e;       // weight rows per expert (F for MODE 0, d for MODE 1)
    int splits;           // S
    int kb_per_split;     // K / 64 / S
    const float* scale0;  // row scales of W1 (MODE 0) or W2 (MODE 1), [n][rows_per_e]
    const float* scale1;  // row scales of W3 (MODE 0)
    float* Pa;            // [S][R][ld] partial sums (MODE 1: the only output)
    float* Pb;            // [S][R][ld] (MODE 0 only)
    int R;
    int ld;               // output features (F for MODE 0, d for MODE 1)
    KStatus st;
};

// bf16x2 product, round to nearest (exact for the widened e4m3 values).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Four e4m3 bytes (element order: low byte first) -> four bf16 in two words.
// With the whole bytes at bytes 1 and 3 (f = b0 << 8 | b1 << 24) and the
// magnitudes at bytes 0 and 2 (m = (b0 & 0x7f) | (b1 & 0x7f) << 16),
// f - 240 m = (b0 & 0x80) << 8 | (b0 & 0x7f) << 4 | (the same for b1) << 16:
// each sign at bit 15, each magnitude at bits 4..10, no borrow between the
// halves (checked for all byte pairs) -- one multiply-add instead of a mask,
// a shift and an OR.
__device__ __forceinline__ void widen_e4m3x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    constexpr uint32_t kTwo120 = 0x7B807B80u;   // bf16 2^120 in both halves
    const uint32_t mag = w & 0x7F7F7F7Fu;
    const uint32_t m01 = __byte_perm(mag, 0u, 0x4140), f01 = __byte_perm(w, 0u, 0x1404);
    const uint32_t m23 = __byte_perm(mag, 0u, 0x4342), f23 = __byte_perm(w, 0u, 0x3424);
    lo = mul_bf16x2(f01 - 240u * m01, kTwo120);
    hi = mul_bf16x2(f23 - 240u * m23, kTwo120);
}

__device__ __forceinline__ void widen_chunk(const uint4& v, uint32_t* o) {
    widen_e4m3x4(v.x, o[0], o[1]);
    widen_e4m3x4(v.y, o[2], o[3]);
    widen_e4m3x4(v.z, o[4], o[5]);
    widen_e4m3x4(v.w, o[6], o[7]);
}

template <int MODE>
__global__ void __launch_bounds__(Q8_THREADS, 1)
    tc_decode_fp8_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                         const __grid_constant__ CUtensorMap tmB, Fp8DecArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t ring_u32 = (raw_u32 + 1023u) & ~1023u;
    const uint8_t* ring_ptr = smem_raw + (ring_u32 - raw_u32);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (ring_u32 - raw_u32) + Q8_RING_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Q8_NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_cmax = reinterpret_cast<int*>(tmem_slot + 2);
    int* s_sched = reinterpret_cast<int*>(tmem_slot + 8);
    int* s_touched = s_sched + 3 * Q8_MAX_EXPERTS + 2;

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (Q8_MAX_STAGES + s); };
    auto afull_bar = [&](int s) { return bar0 + 8u * (2 * Q8_MAX_STAGES + s); };
    auto aempty_bar = [&](int s) { return bar0 + 8u * (2 * Q8_MAX_STAGES + Q8_MAX_ASTAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * Q8_MAX_STAGES + 2 * Q8_MAX_ASTAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * Q8_MAX_STAGES + 2 * Q8_MAX_ASTAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * Q8_MAX_STAGES + 2 * Q8_MAX_ASTAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = p.n;
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < Q8_MAX_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), Q8_CONV_WARPS + 1);   // converter warps + the MMA commit
        }
        for (int s = 0; s < Q8_MAX_ASTAGES; ++s) {
            mbar_init(afull_bar(s), Q8_CONV_WARPS);
            mbar_init(aempty_bar(s), 1);
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
        int nt = 0, cmax = 0;
        for (int e = 0; e < n; ++e) {
            if (s_sched[e] > 0) s_touched[nt++] = e;
            cmax = max(cmax, s_sched[e]);
        }
        s_touched[Q8_MAX_EXPERTS - 1] = nt;   // count kept in the last slot (n <= 31)
        *s_cmax = cmax;
    }
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int* counts = s_sched;
    const int* offsets = s_sched + n;
    const int n_touched = s_touched[Q8_MAX_EXPERTS - 1];
    const KStatus st = p.st;

    // Layout for this call, from the largest token count nm (rounded up to 32):
    // ta weight tiles per item (W1 and W3 together while their accumulators fit),
    // acc_sets accumulator sets of ta * nm columns, then A stages of ta * 32
    // columns (64 bf16 per row); the shared ring holds stages of ta fp8 tiles
    // plus nm token rows.  For nm <= 256 this leaves >= 3 A stages and >= 5
    // shared stages.
    const int nm = max(Q8_B_BOX, (*s_cmax + Q8_B_BOX - 1) / Q8_B_BOX * Q8_B_BOX);
    const int ta = (MODE == 0 && nm <= 128) ? 2 : 1;
    const int tsplit = MODE == 0 ? 2 / ta : 1;
    const int acc_stride = ta * nm;
    const int acc_sets = 2 * acc_stride <= 320 ? 2 : 1;
    const int a_col0 = acc_sets * acc_stride;
    const int a_cols = ta * 32;
    const int AS = min(Q8_MAX_ASTAGES, (Q8_TMEM_COLS - Q8_TMEM_SPARE - a_col0) / a_cols);
    const int stage_bytes = ta * Q8_F8_BYTES + nm * Q8_BK * 2;
    const int FS = min(Q8_MAX_STAGES, Q8_RING_BYTES / stage_bytes);
    const int items = n_touched * tsplit * p.row_blocks * p.splits;

    // item -> (expert, weight tile when W1 and W3 run apart, row block, K split)
    auto decode_item = [&](int it, int& e, int& tile, int& rb, int& sp) {
        sp = it % p.splits;
        int r = it / p.splits;
        tile = r % tsplit;
        r /= tsplit;
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
                int e, tile, rb, sp;
                decode_item(it, e, tile, rb, sp);
                const int nbox = item_n(e) / Q8_B_BOX;
                const int arow = e * p.rows_per_e + rb * 128;
                const int brow = offsets[e];
                const uint32_t bytes = ta * Q8_F8_BYTES + nbox * Q8_B_BOX * Q8_BK * 2;
                const CUtensorMap* one = tile == 0 ? &tmA0 : &tmA1;
                for (int kb = sp * p.kb_per_split; kb < (sp + 1) * p.kb_per_split; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, st, abort_flag)) { ok = false; break; }
                    const uint32_t dst = ring_u32 + static_cast<uint32_t>(stage * stage_bytes);
                    mbar_arrive_expect_tx(full_bar(stage), bytes);
                    if (ta == 2) {
                        tma_load_2d(dst, &tmA0, full_bar(stage), kb * Q8_BK, arow, pol_w);
                        tma_load_2d(dst + Q8_F8_BYTES, &tmA1, full_bar(stage), kb * Q8_BK, arow, pol_w);
                    } else {
                        tma_load_2d(dst, one, full_bar(stage), kb * Q8_BK, arow, pol_w);
                    }
                    const uint32_t tok = dst + ta * Q8_F8_BYTES;
                    for (int bb = 0; bb < nbox; ++bb)
                        tma_load_2d(tok + bb * Q8_B_BOX * Q8_BK * 2, &tmB, full_bar(stage), kb * Q8_BK,
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
        // ---------------- converters: fp8 rows -> bf16 A stages in tensor memory ----------------
        // Thread = weight row r of the tile (= tensor-memory lane r).  With two
        // tiles per stage, warp j of a quadrant widens 32 K of tile j/2; with
        // one, 16 K.  The 64-byte swizzle puts 16-byte chunk c of row r at
        // c ^ ((r / 2) % 4), so the eight rows a quarter-warp reads fall in
        // eight different bank groups.
        const int q = warp & 3;
        const int j = (warp - Q8_CONV_WARP0) >> 2;
        const int r = q * 32 + lane;
        const int rsw = (r >> 1) & 3;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        int stage = 0, ast = 0;
        uint32_t phase = 0, aph = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
            for (int k = 0; k < p.kb_per_split; ++k) {
                if (!mbar_wait_warp(full_bar(stage), phase, st, abort_flag)) { ok = false; break; }
                if (!mbar_wait_warp(aempty_bar(ast), aph ^ 1u, st, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint8_t* src = ring_ptr + stage * stage_bytes;
                const uint32_t acol = static_cast<uint32_t>(a_col0 + ast * a_cols);
                if (ta == 2) {
                    const int t = j >> 1, c0 = 2 * (j & 1);
                    const uint8_t* row = src + t * Q8_F8_BYTES + r * Q8_BK;
                    const uint4 v0 = *reinterpret_cast<const uint4*>(row + ((c0 ^ rsw) << 4));
                    const uint4 v1 = *reinterpret_cast<const uint4*>(row + (((c0 + 1) ^ rsw) << 4));
                    uint32_t o[16];
                    widen_chunk(v0, o);
                    widen_chunk(v1, o + 8);
                    tmem_st_32x32b_x16(lane_base + acol + static_cast<uint32_t>(t * 32 + (j & 1) * 16), o);
                } else {
                    const uint8_t* row = src + r * Q8_BK;
                    const uint4 v = *reinterpret_cast<const uint4*>(row + ((j ^ rsw) << 4));
                    uint32_t o[8];
                    widen_chunk(v, o);
                    tmem_st_32x32b_x8(lane_base + acol + static_cast<uint32_t>(j * 8), o);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(empty_bar(stage));
                    mbar_arrive(afull_bar(ast));
                }
                if (++stage == FS) { stage = 0; phase ^= 1u; }
                if (++ast == AS) { ast = 0; aph ^= 1u; }
            }
        }
        if (!ok) {
            if (lane == 0) report(st, kStatusTimeout);
            *abort_flag = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0, ast = 0;
            uint32_t phase = 0, aph = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                int e, tile, rb, sp;
                decode_item(it, e, tile, rb, sp);
                const int N = item_n(e);
                const uint32_t idesc = idesc_bf16_f32(128, N);
                if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, st, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * acc_stride);
                for (int k = 0; k < p.kb_per_split; ++k) {
                    // The converters arrive on afull only after they saw this stage's
                    // full barrier complete, so the token rows' TMA has landed too.
                    if (!mbar_wait(afull_bar(ast), aph, st, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a0 = tmem_base + static_cast<uint32_t>(a_col0 + ast * a_cols);
                    const uint64_t bdesc =
                        sdesc_kmajor_sw128(ring_u32 + static_cast<uint32_t>(stage * stage_bytes + ta * Q8_F8_BYTES));
#pragma unroll
                    for (int kk = 0; kk < Q8_BK / Q8_UMMA_K; ++kk) {
                        const uint32_t accum = (k | kk) != 0;
                        mma_bf16_ts(d0, a0 + 8u * kk, bdesc + 2u * kk, idesc, accum);
                        if (ta == 2) mma_bf16_ts(d0 + nm, a0 + 32u + 8u * kk, bdesc + 2u * kk, idesc, accum);
                    }
                    mma_commit(aempty_bar(ast));
                    mma_commit(empty_bar(stage));
                    if (++stage == FS) { stage = 0; phase ^= 1u; }
                    if (++ast == AS) { ast = 0; aph ^= 1u; }
                }
                if (!ok) break;
                mma_commit(accf_bar(acc));
                if (++acc == acc_sets) {
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
            int e, tile, rb, sp;
            decode_item(it, e, tile, rb, sp);
            const int N = item_n(e);
            const int cnt = counts[e];
            const int off = offsets[e];
            const int feat = rb * 128 + q * 32 + lane;   // this thread's weight row = output feature
            const size_t srow = static_cast<size_t>(e) * p.rows_per_e + feat;
            if (!mbar_wait_warp(accf_bar(acc), acc_phase, st, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t t0 =
                tmem_base + static_cast<uint32_t>(acc * acc_stride) + (static_cast<uint32_t>(q * 32) << 16);
            for (int part = 0; part < ta; ++part) {
                const int tl = ta == 2 ? part : tile;
                const float sc = __ldg((tl == 0 ? p.scale0 : p.scale1) + srow);
                float* P = (tl == 0 ? p.Pa : p.Pb) + static_cast<size_t>(sp) * p.R * p.ld;
                const uint32_t tp = t0 + static_cast<uint32_t>(part * nm);
                for (int c = 0; c < N; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tp + c, v);
                    tmem_ld_wait();
                    const int jn = min(32, cnt - c);
                    float* dst = P + static_cast<size_t>(off + c) * p.ld + feat;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        if (jj < jn) dst[static_cast<size_t>(jj) * p.ld] = sc * __uint_as_float(v[jj]);
                }
            }
            tc_fence_before();
            mbar_arrive(acce_bar(acc));
            if (++acc == acc_sets) {
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

namespace {
template <int MODE>
cudaError_t launch_fp8(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b, Fp8DecArgs args,
                       int num_sms, cudaStream_t s) {
    auto kern = tc_decode_fp8_kernel<MODE>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Q8_SMEM_BYTES));
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(num_sms), dim3(Q8_THREADS), Q8_SMEM_BYTES, s, a0, a1, b, args);
}
}  // namespace

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
