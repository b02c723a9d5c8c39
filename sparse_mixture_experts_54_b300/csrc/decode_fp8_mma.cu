// decode_fp8_mma.cu -- the weight-streaming expert GEMMs with fp8 (e4m3)
// expert weights multiplied directly by the 8-bit tensor-core MMA
// (tcgen05.mma kind::f8f6f4), for the small batches whose layer time is the
// time to stream the touched experts' weights (the memory-vs-compute remark of
// the xyznot summary, "Limitations").
//
// A weight is w = s_w * q: q an e4m3 byte, s_w one fp32 scale per weight row.
// The e4m3 MMA needs both operands in 8 bits, so each bf16 token row v (a
// gathered input row for W1/W3, a SwiGLU row for W2) is written as two e4m3
// rows: with a power-of-two row scale s_v that maps max|v| into (224, 448],
//
//     s_v * v = hi + lo,   hi = e4m3(s_v * v),   lo = e4m3(s_v * v - hi),
//
// exactly for every element with |s_v * v| >= 1/4 (a bf16 value has 8
// significant bits, hi carries the upper 4, lo the rest; below 1/4 the lowest
// bits fall under e4m3's smallest step 2^-9 and are rounded).  The MMA's N
// dimension holds the hi and lo rows of each token side by side (token j ->
// columns 2j, 2j+1), so one pass over the weights gives
//
//     D[f][2j] + D[f][2j+1] = sum_k q[f][k] * s_v[j] * v[j][k]
//
// and the epilogue multiplies by s_w[f] / s_v[j] (exact for power-of-two
// scales).  The products of two e4m3 values are exact; the tensor core sums
// them in fp32.  Compared with widening the weights to bf16 on chip
// (decode_fp8.cu), no integer pipe or tensor-memory store touches the weights:
// they go from HBM by TMA to shared memory and straight into the MMA, with the
// same number of MMA instructions per weight byte as the bf16 kernels of
// decode_tc.cu (K = 32 one-byte elements per instruction instead of 16
// two-byte ones).
//
// Kernels:
//   split_rows_e4m3_kernel       bf16 rows -> hi/lo e4m3 rows + 1/s_v per row;
//   decode_swiglu_split_kernel   the K-split partial sums of W1 and W3 ->
//                                H = bf16(SiLU(a) * b) (as the bf16 path rounds
//                                it) -> hi/lo e4m3 rows + 1/s_v, one scale per
//                                row and per K range of the W2 GEMM's splits;
//   tc_decode_f8_kernel<MODE>    MODE 0: W1/W3 rows x token rows, MODE 1: W2
//                                rows x SwiGLU rows; fp32 partial sums
//                                P[s][row][feature] as decode_tc.cu writes them,
//                                so the SwiGLU and combine steps after them
//                                are unchanged.
//
// Roles of tc_decode_f8_kernel (6 warps, one CTA per SM, persistent over its
// items): warp 0 lane 0 streams weight tiles (128 rows x 128 bytes, 128-byte
// swizzle) and token tiles (hi/lo rows, 32 rows per box) with TMA into a ring
// of stages; warp 1 owns tensor memory and issues the MMAs; warps 2-5 move
// finished accumulators to the partial sums.  The ring depth, whether W1 and
// W3 share an item and the accumulator sets follow the largest per-expert
// token count, read on the device.  Every wait is bounded, as in gemm_tc.cu.
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "kernels.h"

namespace moe {

namespace {
constexpr int F8_BK = 128;                    // K per stage: one 128-byte swizzle row of e4m3
constexpr int F8_UMMA_K = 32;                 // K per kind::f8f6f4 MMA
constexpr int F8_A_BYTES = 128 * F8_BK;       // one 128-row weight tile, 16 KB
constexpr int F8_B_BOX = 32;                  // token rows (hi/lo of 16 tokens) per TMA box
constexpr int F8_THREADS = 192;
constexpr int F8_EPI_THREADS = 128;
constexpr int F8_MAX_EXPERTS = 32;
constexpr int F8_MAX_STAGES = 12;
constexpr int F8_NUM_BARS = 2 * F8_MAX_STAGES + 2 + 2 + 1;
constexpr int F8_TMEM_COLS = 512;
constexpr size_t F8_SMEM_BYTES = 227 * 1024;
constexpr size_t F8_SMEM_FIXED = 1024 + F8_NUM_BARS * 8 + 32 + (3 * F8_MAX_EXPERTS + 2) * 4 + F8_MAX_EXPERTS * 4;
constexpr int F8_RING_BYTES = static_cast<int>((F8_SMEM_BYTES - F8_SMEM_FIXED) / 1024 * 1024);
}  // namespace

// ---------------------------------------------------------------------------
// e4m3 helpers (round to nearest even, saturating to +-448; the hardware
// conversions of PTX cvt)

// Two floats -> two e4m3 bytes; `lo` goes to the low byte (the lower address).
__device__ __forceinline__ uint16_t e4m3x2_from(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// Two e4m3 bytes -> their exact values (every e4m3 value is an f16 value).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t v) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    __half2 h;
    memcpy(&h, &h2, 4);
    return __half22float2(h);   // .x from the low byte
}
// hi/lo bytes of two scaled values: s*v = hi + lo (see the file comment).
__device__ __forceinline__ void split2(float v0, float v1, float s, uint16_t& hi, uint16_t& lo) {
    const float a = v0 * s, b = v1 * s;
    hi = e4m3x2_from(a, b);
    const float2 h = e4m3x2_to_float2(hi);
    lo = e4m3x2_from(a - h.x, b - h.y);
}
// Power-of-two scale s with max*s in (224, 448], and 1/s (max == 0: 1 and 1).
__device__ __forceinline__ void row_scale(float mx, float& s, float& inv) {
    if (!(mx > 0.0f) || !isfinite(mx)) {
        s = 1.0f;
        inv = 1.0f;
        return;
    }
    const uint32_t bits = __float_as_uint(mx);
    const int E = static_cast<int>((bits >> 23) & 0xFF) - 127;
    int k = ((bits & 0x7FFFFFu) <= 0x600000u ? 8 : 7) - E;   // 448 = 1.75 * 2^8
    k = max(-126, min(126, k));
    s = __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
    inv = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------------------
// bf16 rows X [R][d] -> Xq [2R][d] bytes (row 2r: hi, row 2r+1: lo) and
// xinv[r] = 1/s.  One warp per row; d a multiple of 8.
__global__ void __launch_bounds__(256) split_rows_e4m3_kernel(const __nv_bfloat16* __restrict__ X, int R, int d,
                                                              uint8_t* __restrict__ Xq, float* __restrict__ xinv) {
    griddep_launch_dependents();
    griddep_wait();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= R) return;
    const uint4* row = reinterpret_cast<const uint4*>(X + static_cast<size_t>(warp) * d);
    const int nv = d / 8;
    float mx = 0.0f;
    for (int v = lane; v < nv; v += 32) {
        const uint4 u = __ldg(row + v);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
    mx = warp_max(mx);
    float s, inv;
    row_scale(mx, s, inv);
    uint2* hi_row = reinterpret_cast<uint2*>(Xq + static_cast<size_t>(2 * warp) * d);
    uint2* lo_row = reinterpret_cast<uint2*>(Xq + static_cast<size_t>(2 * warp + 1) * d);
    for (int v = lane; v < nv; v += 32) {
        const uint4 u = __ldg(row + v);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
        uint16_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(h[i]);
            split2(f.x, f.y, s, hi[i], lo[i]);
        }
        hi_row[v] = make_uint2(hi[0] | (static_cast<uint32_t>(hi[1]) << 16), hi[2] | (static_cast<uint32_t>(hi[3]) << 16));
        lo_row[v] = make_uint2(lo[0] | (static_cast<uint32_t>(lo[1]) << 16), lo[2] | (static_cast<uint32_t>(lo[3]) << 16));
    }
    if (lane == 0) xinv[warp] = inv;
}

// H row r = bf16(SiLU(sum_s Pa[s][r]) * sum_s Pb[s][r]) (parts added in order,
// as decode_swiglu_kernel does), then split like split_rows_e4m3_kernel into
// Hq rows 2r / 2r+1, with one scale per row and per chunk of `chunk` features:
// chunk c is exactly the K range of the W2 GEMM's split c, within which the
// scale has to be constant; hinv[c][r] = 1/s.  Block (c, r) does chunk c of
// row r; chunk a multiple of 8.
__global__ void __launch_bounds__(256, 2) decode_swiglu_split_kernel(const float* __restrict__ Pa,
                                                                  const float* __restrict__ Pb, int S, int R, int F,
                                                                  int chunk, uint8_t* __restrict__ Hq,
                                                                  float* __restrict__ hinv) {
    extern __shared__ float hs_row[];   // [chunk]: this chunk's bf16 values
    __shared__ float s_max[8];
    griddep_launch_dependents();
    griddep_wait();
    const int c = blockIdx.x, r = blockIdx.y;
    const size_t base = static_cast<size_t>(r) * F + static_cast<size_t>(c) * chunk;
    const size_t part4 = static_cast<size_t>(R) * F / 4;
    const float4* pa = reinterpret_cast<const float4*>(Pa + base);
    const float4* pb = reinterpret_cast<const float4*>(Pb + base);
    float mx = 0.0f;
    for (int i = threadIdx.x; i < chunk / 4; i += blockDim.x) {
        const float4 a = sum_splits(pa + i, part4, S), b = sum_splits(pb + i, part4, S);
        float h[4] = {silu_f(a.x) * b.x, silu_f(a.y) * b.y, silu_f(a.z) * b.z, silu_f(a.w) * b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            h[j] = __bfloat162float(__float2bfloat16_rn(h[j]));
            mx = fmaxf(mx, fabsf(h[j]));
        }
        reinterpret_cast<float4*>(hs_row)[i] = make_float4(h[0], h[1], h[2], h[3]);
    }
    mx = warp_max(mx);
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x < 32) {
        float m = threadIdx.x < (blockDim.x >> 5) ? s_max[threadIdx.x] : 0.0f;
        m = warp_max(m);
        if (threadIdx.x == 0) s_max[0] = m;
    }
    __syncthreads();
    float s, inv;
    row_scale(s_max[0], s, inv);
    uint2* hi_row = reinterpret_cast<uint2*>(Hq + static_cast<size_t>(2 * r) * F + static_cast<size_t>(c) * chunk);
    uint2* lo_row = reinterpret_cast<uint2*>(Hq + static_cast<size_t>(2 * r + 1) * F + static_cast<size_t>(c) * chunk);
    for (int i = threadIdx.x; i < chunk / 8; i += blockDim.x) {
        const float4 a = reinterpret_cast<const float4*>(hs_row)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(hs_row)[2 * i + 1];
        uint16_t hi[4], lo[4];
        split2(a.x, a.y, s, hi[0], lo[0]);
        split2(a.z, a.w, s, hi[1], lo[1]);
        split2(b.x, b.y, s, hi[2], lo[2]);
        split2(b.z, b.w, s, hi[3], lo[3]);
        hi_row[i] = make_uint2(hi[0] | (static_cast<uint32_t>(hi[1]) << 16), hi[2] | (static_cast<uint32_t>(hi[3]) << 16));
        lo_row[i] = make_uint2(lo[0] | (static_cast<uint32_t>(lo[1]) << 16), lo[2] | (static_cast<uint32_t>(lo[3]) << 16));
    }
    if (threadIdx.x == 0) hinv[static_cast<size_t>(c) * R + r] = inv;
}

// ---------------------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]^T, e4m3 inputs, fp32 accumulator, one CTA.
__device__ __forceinline__ void mma_e4m3_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Instruction descriptor, kind::f8f6f4: e4m3 A and B (both K-major), fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4)                                   // D format: f32
           | (0u << 7)                                 // A format: e4m3
           | (0u << 10)                                // B format: e4m3
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

struct F8DecArgs {
    const int* sched;
    int n;
    int row_blocks;       // weight rows per expert / 128
    int rows_per_e;       // weight rows per expert (F for MODE 0, d for MODE 1)
    int splits;           // S
    int kb_per_split;     // K / 128 / S
    const float* scale0;  // row scales of W1 (MODE 0) or W2 (MODE 1), [n][rows_per_e]
    const float* scale1;  // row scales of W3 (MODE 0)
    const float* vinv;    // 1/s_v of the token rows: [R] (MODE 0) or [S][R] (MODE 1, one per K split)
    int vinv_split;       // stride of vinv between K splits (0: one scale per row)
    float* Pa;            // [S][R][ld] partial sums (MODE 1: the only output)
    float* Pb;            // [S][R][ld] (MODE 0 only)
    int R;
    int ld;               // output features (F for MODE 0, d for MODE 1)
    KStatus st;
};

template <int MODE>
__global__ void __launch_bounds__(F8_THREADS, 1)
    tc_decode_f8_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB, F8DecArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t ring_u32 = (raw_u32 + 1023u) & ~1023u;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (ring_u32 - raw_u32) + F8_RING_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + F8_NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* s_cmax = reinterpret_cast<int*>(tmem_slot + 2);
    int* s_sched = reinterpret_cast<int*>(tmem_slot + 8);
    int* s_touched = s_sched + 3 * F8_MAX_EXPERTS + 2;

    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (F8_MAX_STAGES + s); };
    auto accf_bar = [&](int b) { return bar0 + 8u * (2 * F8_MAX_STAGES + b); };
    auto acce_bar = [&](int b) { return bar0 + 8u * (2 * F8_MAX_STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * F8_MAX_STAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = p.n;
    griddep_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < F8_MAX_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), F8_EPI_THREADS);
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
        tmem_alloc(smem_u32(tmem_slot), F8_TMEM_COLS);
        tmem_relinquish();
    }
    // Nothing above reads a buffer of the layer; the schedule, the token rows
    // and their scales come from the kernels before this one.
    griddep_wait();
    for (int i = threadIdx.x; i < 3 * n + 2; i += F8_THREADS) s_sched[i] = p.sched[i];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        int nt = 0, cmax = 0;
        for (int e = 0; e < n; ++e) {
            if (s_sched[e] > 0) s_touched[nt++] = e;
            cmax = max(cmax, s_sched[e]);
        }
        s_touched[F8_MAX_EXPERTS - 1] = nt;   // count kept in the last slot (n <= 31)
        *s_cmax = cmax;
    }
    __syncthreads();
    const uint32_t tmem_base = *tmem_slot;
    const int* counts = s_sched;
    const int* offsets = s_sched + n;
    const int n_touched = s_touched[F8_MAX_EXPERTS - 1];
    const KStatus st = p.st;

    // Layout for this call, from the largest token count nm (rounded up to 16,
    // at most 256): W1 and W3 share an item (ta = 2 weight tiles per stage)
    // while nm <= 64; an accumulator holds ta * 2nm columns (hi and lo of each
    // token), two sets when they fit in the 512 columns; a stage holds ta
    // weight tiles and 2nm token rows of 128 bytes.
    const int nm = max(16, (*s_cmax + 15) / 16 * 16);
    const int ta = (MODE == 0 && nm <= 64) ? 2 : 1;
    const int tsplit = MODE == 0 ? 2 / ta : 1;
    const int acc_stride = ta * 2 * nm;
    const int acc_sets = 2 * acc_stride <= F8_TMEM_COLS ? 2 : 1;
    const int stage_bytes = ta * F8_A_BYTES + 2 * nm * F8_BK;
    const int FS = min(F8_MAX_STAGES, F8_RING_BYTES / stage_bytes);
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
    // tokens of an expert rounded up to 16 (the MMA covers 2x that many rows; 16
    // rather than 32 measured ~1.4% faster at T = 1..128: smaller MMAs and stages)
    auto item_n = [&](int e) { return max(16, (counts[e] + 15) / 16 * 16); };

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
                const int nbox = item_n(e) / 16;   // 32 hi/lo rows per box
                const int arow = e * p.rows_per_e + rb * 128;
                const int brow = 2 * offsets[e];
                const uint32_t bytes = ta * F8_A_BYTES + nbox * F8_B_BOX * F8_BK;
                const CUtensorMap* one = tile == 0 ? &tmA0 : &tmA1;
                for (int kb = sp * p.kb_per_split; kb < (sp + 1) * p.kb_per_split; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, st, abort_flag)) { ok = false; break; }
                    const uint32_t dst = ring_u32 + static_cast<uint32_t>(stage * stage_bytes);
                    mbar_arrive_expect_tx(full_bar(stage), bytes);
                    if (ta == 2) {
                        tma_load_2d(dst, &tmA0, full_bar(stage), kb * F8_BK, arow, pol_w);
                        tma_load_2d(dst + F8_A_BYTES, &tmA1, full_bar(stage), kb * F8_BK, arow, pol_w);
                    } else {
                        tma_load_2d(dst, one, full_bar(stage), kb * F8_BK, arow, pol_w);
                    }
                    const uint32_t tok = dst + ta * F8_A_BYTES;
                    for (int bb = 0; bb < nbox; ++bb)
                        tma_load_2d(tok + bb * F8_B_BOX * F8_BK, &tmB, full_bar(stage), kb * F8_BK,
                                    brow + bb * F8_B_BOX, pol_x);
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
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < items && ok; it += gridDim.x) {
                int e, tile, rb, sp;
                decode_item(it, e, tile, rb, sp);
                const int N2 = 2 * item_n(e);               // MMA columns of this item
                const int nh = N2 <= 256 ? 1 : 2;           // N > 256: two MMAs of N2/2
                const int Nm = N2 / nh;
                const uint32_t idesc = idesc_e4m3_f32(128, Nm);
                if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, st, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * acc_stride);
                for (int k = 0; k < p.kb_per_split; ++k) {
                    if (!mbar_wait(full_bar(stage), phase, st, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = ring_u32 + static_cast<uint32_t>(stage * stage_bytes);
                    const uint32_t b_addr = a_addr + ta * F8_A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < F8_BK / F8_UMMA_K; ++kk) {
                        const uint32_t accum = (k | kk) != 0;
                        for (int t = 0; t < ta; ++t) {
                            const uint64_t adesc = sdesc_kmajor_sw128(a_addr + t * F8_A_BYTES) + 2u * kk;
                            for (int h = 0; h < nh; ++h) {
                                const uint64_t bdesc = sdesc_kmajor_sw128(b_addr + h * Nm * F8_BK) + 2u * kk;
                                mma_e4m3_ss(d0 + static_cast<uint32_t>(t * 2 * nm + h * Nm), adesc, bdesc, idesc,
                                            accum);
                            }
                        }
                    }
                    mma_commit(empty_bar(stage));
                    if (++stage == FS) { stage = 0; phase ^= 1u; }
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
        // ---------------- epilogue: (hi + lo) x s_w / s_v -> fp32 partial sums ----------------
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < items; it += gridDim.x) {
            int e, tile, rb, sp;
            decode_item(it, e, tile, rb, sp);
            const int N2 = 2 * item_n(e);
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
                const float sw = __ldg((tl == 0 ? p.scale0 : p.scale1) + srow);
                float* P = (tl == 0 ? p.Pa : p.Pb) + static_cast<size_t>(sp) * p.R * p.ld;
                const uint32_t tp = t0 + static_cast<uint32_t>(part * 2 * nm);
                for (int c2 = 0; c2 < N2; c2 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tp + c2, v);
                    tmem_ld_wait();
                    const int tok0 = c2 / 2;
                    // 1/s_v of the 16 tokens of these columns, one per lane, then broadcast
                    const float* vinv = p.vinv + static_cast<size_t>(sp) * p.vinv_split;
                    const float vi_l = (lane < 16 && tok0 + lane < cnt) ? __ldg(vinv + off + tok0 + lane) : 0.0f;
                    float* dst = P + static_cast<size_t>(off + tok0) * p.ld + feat;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float vi = __shfl_sync(0xffffffffu, vi_l, jj);
                        if (tok0 + jj < cnt)
                            dst[static_cast<size_t>(jj) * p.ld] =
                                (__uint_as_float(v[2 * jj]) + __uint_as_float(v[2 * jj + 1])) * sw * vi;
                    }
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
        tmem_dealloc(tmem_base, F8_TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// host side

// Row-major byte matrix [rows][cols] (cols a multiple of 128) -> tensor map
// with a (128-byte x box_rows) box and 128-byte swizzle, the layout of a K-major
// e4m3 MMA operand (rows of 128 one-byte elements, 8-row groups 1024 B apart).
bool encode_map_u8_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    if (rows == 0 || cols == 0 || cols % 128) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {
template <int MODE>
cudaError_t launch_f8(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b, F8DecArgs args, int num_sms,
                      cudaStream_t s) {
    auto kern = tc_decode_f8_kernel<MODE>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(F8_SMEM_BYTES));
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(num_sms), dim3(F8_THREADS), F8_SMEM_BYTES, s, a0, a1, b, args);
}
}  // namespace

cudaError_t launch_split_rows_e4m3(const __nv_bfloat16* X, int R, int d, uint8_t* Xq, float* xinv, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    if (d % 8) return cudaErrorInvalidValue;
    const int blocks = (R + 7) / 8;   // 8 warps = 8 rows per block
    return launch_pdl(split_rows_e4m3_kernel, dim3(blocks), dim3(256), 0, s, X, R, d, Xq, xinv);
}

cudaError_t launch_decode_swiglu_split(const float* Pa, const float* Pb, int S, int R, int F, int chunks, uint8_t* Hq,
                                       float* hinv, cudaStream_t s) {
    if (R <= 0) return cudaSuccess;
    if (chunks < 1 || F % chunks || (F / chunks) % 8) return cudaErrorInvalidValue;
    const int chunk = F / chunks;
    const size_t smem = static_cast<size_t>(chunk) * 4;
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    cudaError_t err = cudaFuncSetAttribute(decode_swiglu_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(decode_swiglu_split_kernel, dim3(chunks, R), dim3(256), smem, s, Pa, Pb, S, R, F, chunk, Hq,
                      hinv);
}

cudaError_t launch_decode_f8_w13(const CUtensorMap& mapW1q, const CUtensorMap& mapW3q, const CUtensorMap& mapXq,
                                 const float* W1s, const float* W3s, const float* xinv, const int* sched, int n, int d,
                                 int F, int T, int K, int splits, float* Pa, float* Pb, KStatus st, int num_sms,
                                 cudaStream_t s) {
    if (n > F8_MAX_EXPERTS - 1 || T <= 0 || T > kDecodeMaxT || d % F8_BK || F % 128) return cudaErrorInvalidValue;
    F8DecArgs args{};
    args.sched = sched;
    args.n = n;
    args.row_blocks = F / 128;
    args.rows_per_e = F;
    args.splits = splits;
    args.kb_per_split = d / F8_BK / splits;
    args.scale0 = W1s;
    args.scale1 = W3s;
    args.vinv = xinv;
    args.vinv_split = 0;
    args.Pa = Pa;
    args.Pb = Pb;
    args.R = K * T;
    args.ld = F;
    args.st = st;
    return launch_f8<0>(mapW1q, mapW3q, mapXq, args, num_sms, s);
}

cudaError_t launch_decode_f8_w2(const CUtensorMap& mapW2q, const CUtensorMap& mapHq, const float* W2s,
                                const float* hinv, const int* sched, int n, int d, int F, int T, int K, int splits,
                                float* P2, KStatus st, int num_sms, cudaStream_t s) {
    if (n > F8_MAX_EXPERTS - 1 || T <= 0 || T > kDecodeMaxT || F % F8_BK || d % 128) return cudaErrorInvalidValue;
    F8DecArgs args{};
    args.sched = sched;
    args.n = n;
    args.row_blocks = d / 128;
    args.rows_per_e = d;
    args.splits = splits;
    args.kb_per_split = F / F8_BK / splits;
    args.scale0 = W2s;
    args.scale1 = W2s;
    args.vinv = hinv;
    args.vinv_split = K * T;
    args.Pa = P2;
    args.Pb = nullptr;
    args.R = K * T;
    args.ld = d;
    args.st = st;
    return launch_f8<1>(mapW2q, mapW2q, mapHq, args, num_sms, s);
}

}  // namespace moe
